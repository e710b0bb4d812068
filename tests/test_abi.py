"""Host-only checks of the C ABI: the library builds, loads, exports every declared
entry point, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as m
    return m._load()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(mla_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("mla_get_metadata", "mla_decode_fwd", "mla_metadata_shape",
                 "mla_workspace_size", "mla_get_device_error", "mla_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"


def test_params_struct_matches(lib):
    import mla_decode_gb300 as m
    assert lib.mla_fwd_params_size() == ctypes.sizeof(m.FwdParams)
    assert lib.mla_abi_version() == m.ABI_VERSION == 5


def test_status_strings(lib):
    import mla_decode_gb300 as m
    for code in range(0, -11, -1):
        s = m.mla_status_string(code)
        assert s and s != "unknown status"
    assert m.mla_status_string(12345) == "unknown status"


def test_metadata_shape(lib):
    import mla_decode_gb300 as m
    assert m.mla_metadata_shape(64, 128, 152) == (76, 8)
    assert m.mla_metadata_shape(64, 16, 152) == (76, 8)
    assert m.mla_metadata_shape(64, 256, 152) == (38, 8)
    assert m.mla_metadata_shape(1, 128, 1) == (1, 8)
    with pytest.raises(m.MlaError):
        m.mla_metadata_shape(0, 128, 152)
    with pytest.raises(m.MlaError):
        m.mla_metadata_shape(4, 0, 152)
    # the scheduler evaluates at most 512 part counts: num_sm is bounded
    assert m.mla_metadata_shape(4, 128, m.MAX_NUM_SM) == (m.MAX_NUM_SM // 2, 8)
    with pytest.raises(m.MlaError):
        m.mla_metadata_shape(4, 128, m.MAX_NUM_SM + 1)


def test_workspace_size(lib):
    import mla_decode_gb300 as m
    n = m.mla_workspace_size(64, 128, 76)
    splits = 64 + 76
    # partials, LSEs (padded to 256 bytes), then the fused combine's two 8-byte
    # barrier counters in a 256-byte tail
    assert n >= splits * 128 * 512 * 4 + splits * 128 * 4 + 16
    assert n < splits * 128 * 512 * 4 + splits * 128 * 4 + 768


def good_params():
    import mla_decode_gb300 as m
    p = m.FwdParams()
    fake = 1 << 20  # aligned, never dereferenced: validation fails first
    p.b, p.seqlen_q, p.h, p.h_k, p.d, p.d_v, p.dtype = 2, 1, 16, 1, 576, 512, 1
    p.softmax_scale = 0.1
    p.q, p.q_batch_stride, p.q_head_stride = fake, 16 * 576, 576
    p.kv_cache, p.kv_page_stride, p.kv_row_stride = fake, 64 * 576, 576
    p.num_pages, p.page_block_size = 4, 64
    p.block_table, p.block_table_batch_stride, p.max_blocks_per_seq = fake, 2, 2
    p.cache_seqlens = fake
    p.out, p.o_batch_stride, p.o_head_stride = fake, 16 * 512, 512
    p.lse, p.lse_batch_stride = fake, 16
    p.tile_scheduler_metadata, p.num_splits, p.num_sm_parts = fake, fake, 1
    p.workspace = fake
    p.workspace_bytes = m.mla_workspace_size(2, 16, 1)
    return p


@pytest.mark.parametrize("field,value,code", [
    ("q", 0, -1), ("kv_cache", 0, -1), ("workspace", 0, -1), ("lse", 0, -1),
    ("seqlen_q", 0, -2), ("seqlen_q", 2, -2), ("h_k", 2, -2), ("d", 512, -2), ("d_v", 576, -2), ("h", 0, -2),
    ("b", 0, -2), ("dtype", 7, -3), ("page_block_size", 96, -5), ("page_block_size", 0, -5),
    ("q", (1 << 20) + 8, -4), ("q_head_stride", 580, -4), ("kv_page_stride", 64 * 576 + 4, -4),
    ("workspace_bytes", 100, -6), ("num_sm_parts", 0, -2), ("lse_batch_stride", 8, -2),
    ("kv_row_stride", 512, -2), ("max_blocks_per_seq", 0, -2),
])
def test_validation_rejects(lib, field, value, code):
    p = good_params()
    setattr(p, field, value)
    assert lib.mla_decode_fwd(ctypes.byref(p), None) == code


SEP_K = {"k_pe": (1 << 20) + 4096, "k_pe_page_stride": 64 * 64, "k_pe_row_stride": 64,
         "kv_row_stride": 512, "kv_page_stride": 64 * 512}
SEP_Q = {"q_pe": (1 << 20) + 8192, "q_pe_batch_stride": 16 * 64, "q_pe_head_stride": 64}


@pytest.mark.parametrize("fields,code", [
    ({**SEP_K, "k_pe_row_stride": 32}, -2),                 # row narrower than 64 columns
    ({**SEP_K, "k_pe_page_stride": 64 * 64 - 8}, -2),       # page shorter than its rows
    ({**SEP_K, "kv_row_stride": 504, "kv_page_stride": 64 * 504}, -2),
    ({**SEP_K, "k_pe": (1 << 20) + 4104}, -4),              # 8-byte aligned only
    ({**SEP_K, "k_pe_row_stride": 68, "k_pe_page_stride": 64 * 68}, -4),
    ({**SEP_Q, "q_pe_head_stride": 0}, -2),
    ({**SEP_Q, "q_pe_batch_stride": 16 * 64 + 4}, -4),
    ({**SEP_Q, "q_pe": (1 << 20) + 8200}, -4),
    ({"kv_row_stride": 512, "kv_page_stride": 64 * 512}, -2),  # 512-wide rows need k_pe
])
def test_split_layout_rejects(lib, fields, code):
    """Q / Q_pe and KV / K_pe as separate tensors: the same host-side checks."""
    p = good_params()
    for k, v in fields.items():
        setattr(p, k, v)
    assert lib.mla_decode_fwd(ctypes.byref(p), None) == code


@pytest.mark.parametrize("fields,code", [
    ({"seqlen_q": 2}, -2),                                   # lse rows: 16 < 2 * 16
    ({"seqlen_q": 65, "lse_batch_stride": 65 * 16}, -2),     # 1040 query rows > 1024
    ({"seqlen_q": 2, "lse_batch_stride": 32}, -6),           # workspace sized for 16 rows
    ({"seqlen_q": -1}, -2),
])
def test_query_tokens_rejects(lib, fields, code):
    """seqlen_q > 1: rows = seqlen_q * h size lse and the workspace; at most 1024 rows."""
    p = good_params()
    for k, v in fields.items():
        setattr(p, k, v)
    assert lib.mla_decode_fwd(ctypes.byref(p), None) == code


def e4m3_params():
    p = good_params()
    p.dtype, p.q_scale, p.kv_scale = 2, 0.5, 2.0
    return p


@pytest.mark.parametrize("fields,code", [
    ({}, -6),                                                  # valid up to the (small) workspace
    ({"q_scale": 0.0}, -3), ({"kv_scale": -1.0}, -3),
    ({"q_scale": float("nan")}, -3), ({"kv_scale": float("inf")}, -3),
    ({**SEP_K}, -3), ({**SEP_Q}, -3),                          # fused layout only
    ({"q_head_stride": 584}, -4),                              # 8 bytes: not a multiple of 16
    ({"kv_row_stride": 584, "kv_page_stride": 64 * 584}, -4),
    ({"kv_page_stride": 64 * 576 + 8}, -4),
    ({"o_head_stride": 516}, -4),                              # bf16 out: 8 elements
])
def test_e4m3_validation(lib, fields, code):
    """e4m3: finite positive scales, the fused layout, strides of 16 bytes."""
    p = e4m3_params()
    p.workspace_bytes = 100
    for k, v in fields.items():
        setattr(p, k, v)
    assert lib.mla_decode_fwd(ctypes.byref(p), None) == code


def test_null_params(lib):
    assert lib.mla_decode_fwd(None, None) == -1
