"""Host-side argument checks of the Python binding (no GPU): wrong shapes and dtypes
are refused with a ValueError before anything reaches the C library."""
import pytest
import torch


@pytest.fixture(scope="module")
def mla():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as m
    m._load()
    return m


def tensors(b=2, s=1, h=16, pages=4, page=64, q_cols=576, kv_cols=576, dtype=torch.bfloat16):
    return dict(q=torch.zeros(b, s, h, q_cols, dtype=dtype),
                kv_cache=torch.zeros(pages, page, 1, kv_cols, dtype=dtype),
                block_table=torch.zeros(b, 2, dtype=torch.int32),
                cache_seqlens=torch.zeros(b, dtype=torch.int32),
                tile_scheduler_metadata=torch.zeros(1, 8, dtype=torch.int32),
                num_splits=torch.zeros(b + 1, dtype=torch.int32))


def call(mla, t, **kw):
    return mla.prepare_decode(t["q"], t["kv_cache"], t["block_table"], t["cache_seqlens"], 0.1,
                              t["tile_scheduler_metadata"], t["num_splits"], **kw)


@pytest.mark.parametrize("kw,t_kw,match", [
    ({}, dict(q_cols=512), r"q must be \[b, s, h, 576\]"),
    ({}, dict(kv_cols=512), r"kv_cache must be"),
    ({}, dict(dtype=torch.float32), r"fp16, bf16 or float8_e4m3fn"),
    ({"q_pe": torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16)}, {}, r"q must be \[b, s, h, 512\]"),
    ({"k_pe": torch.zeros(4, 64, 1, 64, dtype=torch.bfloat16)}, {}, r"kv_cache must be .*512"),
])
def test_shape_and_dtype_errors(mla, kw, t_kw, match):
    with pytest.raises(ValueError, match=match):
        call(mla, tensors(**t_kw), **kw)


def test_split_layout_tensor_shapes(mla):
    t = tensors(q_cols=512, kv_cols=512)
    with pytest.raises(ValueError, match=r"q_pe must be \[b, s, h, 64\]"):
        call(mla, t, q_pe=torch.zeros(2, 1, 16, 32, dtype=torch.bfloat16),
             k_pe=torch.zeros(4, 64, 1, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match=r"k_pe must be"):
        call(mla, t, q_pe=torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16),
             k_pe=torch.zeros(4, 32, 1, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match=r"q_pe must have q's dtype"):
        call(mla, t, q_pe=torch.zeros(2, 1, 16, 64, dtype=torch.float16),
             k_pe=torch.zeros(4, 64, 1, 64, dtype=torch.bfloat16))


def test_query_token_shape_of_q_pe(mla):
    # q_pe must carry the same number of query tokens as q
    t = tensors(s=2, q_cols=512)
    with pytest.raises(ValueError, match=r"q_pe must be \[b, s, h, 64\]"):
        call(mla, t, q_pe=torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16))


def test_e4m3_checks(mla):
    t = tensors(dtype=torch.float8_e4m3fn)
    # the e4m3 cache keeps its RoPE columns inside the rows
    with pytest.raises(ValueError, match=r"RoPE columns inside"):
        call(mla, tensors(q_cols=512, dtype=torch.float8_e4m3fn),
             q_pe=torch.zeros(2, 1, 16, 64, dtype=torch.float8_e4m3fn))
    # q and the cache share the dtype
    t["kv_cache"] = torch.zeros(4, 64, 1, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"must share dtype"):
        call(mla, t)
    # e4m3 gives bf16 outputs
    assert mla.out_dtype(torch.float8_e4m3fn) == torch.bfloat16
    assert mla.out_dtype(torch.float16) == torch.float16


def test_host_tensors_are_refused(mla):
    # well-formed shapes, but host memory: the binding asks for CUDA tensors
    with pytest.raises(ValueError, match=r"must be on"):
        call(mla, tensors())
