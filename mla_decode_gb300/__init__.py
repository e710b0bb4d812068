"""GB300 (sm_103a) MLA decode: thin Python binding over the library's C ABI.

Every function here has the name of the C entry point it wraps
(include/mla_decode.h) and only marshals arguments: it checks tensor
shapes/dtypes/devices, allocates caller-owned outputs with torch when they are
not given, and passes raw device pointers plus the current CUDA stream.  All
computation happens in the library's CUDA kernels.  If the compiled library is
missing this module raises instead of falling back to anything else; build it
with `python -m mla_decode_gb300._build` (or __graft_entry__.build()).
"""
import ctypes
import os

import torch

from . import _build

__all__ = [
    "MlaError", "mla_abi_version", "mla_status_string", "mla_device_num_sm",
    "mla_metadata_shape", "mla_get_metadata", "mla_workspace_size", "mla_decode_fwd",
    "mla_decode_fwd_timed", "prepare_decode", "DecodeCall", "prepare_metadata", "MetadataCall",
    "mla_get_device_error", "mla_test_forced_timeout", "library_path", "HEAD_DIM", "HEAD_DIM_V", "ROPE_DIM", "BLOCK_N",
    "META_STRIDE", "SCHED_FIXED_COST", "SCHED_SEGMENT_COST", "SCHED_SPLIT_COST", "MAX_NUM_SM", "out_dtype",
]

HEAD_DIM = 576
HEAD_DIM_V = 512
ROPE_DIM = HEAD_DIM - HEAD_DIM_V
ABI_VERSION = 5
BLOCK_N = 64
META_STRIDE = 8
SCHED_FIXED_COST = 5
SCHED_SEGMENT_COST = 16
SCHED_SPLIT_COST = 10
MAX_NUM_SM = 2046
STATIC_WORKSPACE_BYTES = 64 << 20
_DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float8_e4m3fn: 2}


def out_dtype(dtype):
    """dtype of `out` for q / kv_cache of `dtype`: the same, bf16 for e4m3."""
    return torch.bfloat16 if dtype == torch.float8_e4m3fn else dtype


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class MlaError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {mla_status_string(status)} ({status})")


class FwdParams(ctypes.Structure):
    """Mirror of `mla_fwd_params` (checked against the library's sizeof at load)."""
    _fields_ = [
        ("b", _i32), ("seqlen_q", _i32), ("h", _i32), ("h_k", _i32), ("d", _i32),
        ("d_v", _i32), ("dtype", _i32), ("softmax_scale", ctypes.c_float),
        ("q", _vp), ("q_batch_stride", _i64), ("q_head_stride", _i64),
        ("kv_cache", _vp), ("kv_page_stride", _i64), ("kv_row_stride", _i64),
        ("num_pages", _i32), ("page_block_size", _i32),
        ("block_table", _vp), ("block_table_batch_stride", _i64), ("max_blocks_per_seq", _i32),
        ("cache_seqlens", _vp),
        ("out", _vp), ("o_batch_stride", _i64), ("o_head_stride", _i64),
        ("lse", _vp), ("lse_batch_stride", _i64),
        ("tile_scheduler_metadata", _vp), ("num_splits", _vp), ("num_sm_parts", _i32),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("q_pe", _vp), ("q_pe_batch_stride", _i64), ("q_pe_head_stride", _i64),
        ("k_pe", _vp), ("k_pe_page_stride", _i64), ("k_pe_row_stride", _i64),
        ("is_causal", _i32),
        ("q_scale", ctypes.c_float), ("kv_scale", ctypes.c_float),
        ("fused_combine", ctypes.c_int32),
    ]


_lib = None


def library_path():
    return _build.LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise ImportError(
            f"MLA decode library not built ({_build.LIB} missing); "
            "run `python -m mla_decode_gb300._build`")
    lib = ctypes.CDLL(_build.LIB)
    lib.mla_abi_version.restype = ctypes.c_int
    lib.mla_fwd_params_size.restype = ctypes.c_size_t
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_device_num_sm.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.mla_metadata_shape.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.mla_get_metadata.argtypes = [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]
    lib.mla_workspace_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_size_t)]
    lib.mla_decode_fwd.argtypes = [ctypes.POINTER(FwdParams), _vp]
    lib.mla_decode_fwd_timed.argtypes = [ctypes.POINTER(FwdParams), _vp, _vp, _vp]
    lib.mla_decode_fwd_static.argtypes = [ctypes.POINTER(FwdParams), _vp]
    lib.mla_get_device_error.argtypes = [_vp, ctypes.POINTER(ctypes.c_int)]
    lib.mla_test_forced_timeout.argtypes = [ctypes.POINTER(FwdParams), _vp]
    for name in ("mla_device_num_sm", "mla_metadata_shape", "mla_get_metadata",
                 "mla_workspace_size", "mla_decode_fwd", "mla_decode_fwd_timed",
                 "mla_decode_fwd_static", "mla_get_device_error", "mla_test_forced_timeout"):
        getattr(lib, name).restype = ctypes.c_int
    if lib.mla_abi_version() != ABI_VERSION or lib.mla_fwd_params_size() != ctypes.sizeof(FwdParams):
        raise ImportError("MLA decode library ABI mismatch; rebuild it")
    _lib = lib
    return lib


def _check(rc, what):
    if rc != 0:
        raise MlaError(rc, what)


def _stream(device):
    return _vp(torch.cuda.current_stream(device).cuda_stream)


def mla_abi_version():
    return _load().mla_abi_version()


def mla_status_string(status):
    return _load().mla_status_string(int(status)).decode()


def mla_device_num_sm(device=None):
    """SMs the split kernel can occupy at once (2 x co-resident 2-CTA clusters)."""
    dev = torch.cuda.current_device() if device is None else torch.device(device).index or 0
    n = ctypes.c_int(0)
    _check(_load().mla_device_num_sm(int(dev), ctypes.byref(n)), "mla_device_num_sm")
    return n.value


def mla_metadata_shape(b, h, num_sm):
    parts, stride = ctypes.c_int(0), ctypes.c_int(0)
    _check(_load().mla_metadata_shape(int(b), int(h), int(num_sm), ctypes.byref(parts),
                                      ctypes.byref(stride)), "mla_metadata_shape")
    return parts.value, stride.value


def mla_get_metadata(cache_seqlens, h, num_sm=None, tile_scheduler_metadata=None,
                     num_splits=None, seqlen_q=1):
    """Scheduler metadata for `cache_seqlens` (int32 [b], on the GPU), h query heads
    and seqlen_q query tokens per sequence (the C call gets seqlen_q * h rows).

    Returns (tile_scheduler_metadata int32 [num_sm_parts, 8], num_splits int32 [b + 1]),
    writing into the given tensors when they are passed.
    """
    h = int(h) * int(seqlen_q)
    if cache_seqlens.dtype != torch.int32 or not cache_seqlens.is_cuda or cache_seqlens.dim() != 1:
        raise ValueError("cache_seqlens must be a CUDA int32 vector")
    cache_seqlens = cache_seqlens.contiguous()
    dev = cache_seqlens.device
    if num_sm is None:
        num_sm = mla_device_num_sm(dev)
    b = cache_seqlens.numel()
    parts, stride = mla_metadata_shape(b, h, num_sm)
    meta = tile_scheduler_metadata
    if meta is None:
        meta = torch.empty((parts, stride), dtype=torch.int32, device=dev)
    if num_splits is None:
        num_splits = torch.empty((b + 1,), dtype=torch.int32, device=dev)
    if (meta.shape != (parts, stride) or meta.dtype != torch.int32 or not meta.is_contiguous()
            or num_splits.shape != (b + 1,) or num_splits.dtype != torch.int32
            or not num_splits.is_contiguous()):
        raise ValueError("metadata outputs have the wrong shape/dtype")
    with torch.cuda.device(dev):
        _check(_load().mla_get_metadata(_vp(cache_seqlens.data_ptr()), b, int(h), int(num_sm),
                                        _vp(meta.data_ptr()), _vp(num_splits.data_ptr()),
                                        _stream(dev)), "mla_get_metadata")
    return meta, num_splits


class MetadataCall:
    """A validated, pre-marshalled mla_get_metadata call (reusable: re-run it after
    updating cache_seqlens in place)."""

    def __init__(self, cache_seqlens, rows, num_sm, meta, num_splits):
        self._keep = (cache_seqlens, meta, num_splits)
        self.device = cache_seqlens.device
        self._args = (_vp(cache_seqlens.data_ptr()), cache_seqlens.numel(), int(rows),
                      int(num_sm), _vp(meta.data_ptr()), _vp(num_splits.data_ptr()))
        self.meta, self.num_splits = meta, num_splits

    def __call__(self):
        lib = _load()
        with torch.cuda.device(self.device):
            _check(lib.mla_get_metadata(*self._args, _stream(self.device)), "mla_get_metadata")
        return self.meta, self.num_splits


def prepare_metadata(cache_seqlens, h, num_sm=None, tile_scheduler_metadata=None,
                     num_splits=None, seqlen_q=1):
    """mla_get_metadata's checks and output allocation, done once; returns a
    MetadataCall that launches the metadata kernel on the current stream."""
    if cache_seqlens.dtype != torch.int32 or not cache_seqlens.is_cuda or cache_seqlens.dim() != 1:
        raise ValueError("cache_seqlens must be a CUDA int32 vector")
    if not cache_seqlens.is_contiguous():
        raise ValueError("cache_seqlens must be contiguous")
    dev = cache_seqlens.device
    if num_sm is None:
        num_sm = mla_device_num_sm(dev)
    rows = int(h) * int(seqlen_q)
    b = cache_seqlens.numel()
    parts, stride = mla_metadata_shape(b, rows, num_sm)
    meta = tile_scheduler_metadata
    if meta is None:
        meta = torch.empty((parts, stride), dtype=torch.int32, device=dev)
    if num_splits is None:
        num_splits = torch.empty((b + 1,), dtype=torch.int32, device=dev)
    if (meta.shape != (parts, stride) or meta.dtype != torch.int32 or not meta.is_contiguous()
            or meta.device != dev or num_splits.shape != (b + 1,)
            or num_splits.dtype != torch.int32 or not num_splits.is_contiguous()
            or num_splits.device != dev):
        raise ValueError("metadata outputs have the wrong shape/dtype/device")
    return MetadataCall(cache_seqlens, rows, num_sm, meta, num_splits)


def mla_workspace_size(b, h, num_sm_parts):
    n = ctypes.c_size_t(0)
    _check(_load().mla_workspace_size(int(b), int(h), int(num_sm_parts), ctypes.byref(n)),
           "mla_workspace_size")
    return n.value


def mla_decode_fwd(q, kv_cache, block_table, cache_seqlens, softmax_scale,
                   tile_scheduler_metadata, num_splits, out=None, lse=None, workspace=None,
                   split_events=None, q_pe=None, k_pe=None, is_causal=False, q_scale=1.0,
                   kv_scale=1.0, fused_combine=False):
    """Paged split-KV MLA decode (see prepare_decode for the argument contract).

    split_events: optional (begin, end) torch.cuda.Event pair recorded around the
    split kernel (mla_decode_fwd_timed).  Returns (out, lse).
    """
    call = prepare_decode(q, kv_cache, block_table, cache_seqlens, softmax_scale,
                          tile_scheduler_metadata, num_splits, out, lse, workspace,
                          q_pe=q_pe, k_pe=k_pe, is_causal=is_causal, q_scale=q_scale,
                          kv_scale=kv_scale, fused_combine=fused_combine)
    call(split_events=split_events)
    return call.out, call.lse


class DecodeCall:
    """A validated, pre-marshalled mla_decode_fwd call (reusable: the tensors it
    points at are kept alive by this object; re-run it after updating them in place)."""

    def __init__(self, params, tensors, out, lse):
        self.params = params
        self._keep = tensors
        self.out = out
        self.lse = lse
        self.device = out.device

    def __call__(self, split_events=None):
        lib = _load()
        stream = _stream(self.device)
        with torch.cuda.device(self.device):
            if split_events is None:
                rc = lib.mla_decode_fwd(ctypes.byref(self.params), stream)
            else:
                b, e = split_events
                rc = lib.mla_decode_fwd_timed(ctypes.byref(self.params), stream,
                                              _vp(b.cuda_event), _vp(e.cuda_event))
        _check(rc, "mla_decode_fwd")
        return self.out, self.lse


def prepare_decode(q, kv_cache, block_table, cache_seqlens, softmax_scale,
                   tile_scheduler_metadata, num_splits, out=None, lse=None, workspace=None,
                   q_pe=None, k_pe=None, is_causal=False, q_scale=1.0, kv_scale=1.0,
                   fused_combine=False):
    """Paged split-KV MLA decode.

    q [b, 1, h, 576], kv_cache [num_pages, page_size, 1, 576] (fp16 or bf16, same
    dtype), block_table int32 [b, max_blocks], cache_seqlens int32 [b], metadata
    from mla_get_metadata.  Returns (out [b, 1, h, 512] in q's dtype, lse fp32 [b, h]
    natural-log).  Launches on the current stream of q's device.

    FP8 cache: q and kv_cache both torch.float8_e4m3fn with dequantisation scales
    q_scale and kv_scale (the decode runs on q_scale * q and kv_scale * kv); out is
    bf16; the RoPE columns must be inside q and kv_cache (no q_pe / k_pe).

    Split layout: with q_pe [b, s, h, 64] given, q is [b, s, h, 512] (latent
    columns only); with k_pe [num_pages, page_size, 1, 64] given, kv_cache is
    [num_pages, page_size, 1, 512].  The score is then q . kv + q_pe . k_pe.

    Several query tokens: q [b, s, h, 576] with s > 1 (token stride h times the
    head stride), out [b, s, h, 512], lse [b, s, h]; the cache already holds the s
    new tokens, and with is_causal token qi sees the cached tokens
    t < L - (s - 1 - qi).  The metadata must be made with seqlen_q = s.

    fused_combine: the split kernel combines the sequences it split (after a
    grid-wide barrier) instead of a separate combine kernel; same bits either way.
    It saves the combine kernel's launch when nothing is split; when many
    sequences are split the separate kernel (the default) is faster.
    """
    q_cols = HEAD_DIM_V if q_pe is not None else HEAD_DIM
    kv_cols = HEAD_DIM_V if k_pe is not None else HEAD_DIM
    if q.dim() != 4 or q.shape[3] != q_cols:
        raise ValueError(f"q must be [b, s, h, {q_cols}]")
    s_q = q.shape[1]
    if s_q < 1:
        raise ValueError("q needs at least one query token")
    if kv_cache.dim() != 4 or kv_cache.shape[2] != 1 or kv_cache.shape[3] != kv_cols:
        raise ValueError(f"kv_cache must be [num_pages, page_size, 1, {kv_cols}]")
    if q.dtype not in _DTYPE_CODE or kv_cache.dtype != q.dtype:
        raise ValueError("q and kv_cache must share dtype fp16, bf16 or float8_e4m3fn")
    f8 = q.dtype == torch.float8_e4m3fn
    if f8 and (q_pe is not None or k_pe is not None):
        raise ValueError("an e4m3 cache takes the RoPE columns inside q and kv_cache")
    if q_pe is not None and (q_pe.dim() != 4 or tuple(q_pe.shape) != (q.shape[0], s_q,
                                                                       q.shape[2], ROPE_DIM)):
        raise ValueError("q_pe must be [b, s, h, 64]")
    if k_pe is not None and (k_pe.dim() != 4 or tuple(k_pe.shape) != (kv_cache.shape[0],
                                                                       kv_cache.shape[1], 1,
                                                                       ROPE_DIM)):
        raise ValueError("k_pe must be [num_pages, page_size, 1, 64]")
    for name, t in (("q_pe", q_pe), ("k_pe", k_pe)):
        if t is not None and (t.dtype != q.dtype or t.stride(3) != 1):
            raise ValueError(f"{name} must have q's dtype and contiguous columns")
    for name, t in (("q", q), ("kv_cache", kv_cache), ("block_table", block_table),
                    ("cache_seqlens", cache_seqlens), ("tile_scheduler_metadata",
                                                       tile_scheduler_metadata),
                    ("num_splits", num_splits), ("q_pe", q_pe), ("k_pe", k_pe)):
        if t is not None and (not t.is_cuda or t.device != q.device):
            raise ValueError(f"{name} must be on {q.device}")
    if q.stride(3) != 1 or kv_cache.stride(3) != 1:
        raise ValueError("the columns of q and kv_cache must be contiguous")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be int32 [b, max_blocks] with unit column stride")
    if cache_seqlens.dtype != torch.int32 or not cache_seqlens.is_contiguous():
        raise ValueError("cache_seqlens must be a contiguous int32 vector")
    b, _, h, _ = q.shape
    rows = s_q * h
    for name, t in (("q", q), ("q_pe", q_pe)):
        if t is not None and s_q > 1 and t.stride(1) != h * t.stride(2):
            raise ValueError(f"{name}: the s * h query rows must be evenly strided "
                             "(token stride = h * head stride)")
    if block_table.shape[0] != b or cache_seqlens.numel() != b or num_splits.numel() != b + 1:
        raise ValueError("batch size mismatch among q, block_table, cache_seqlens, num_splits")
    parts = tile_scheduler_metadata.shape[0]
    dev = q.device
    lse_shape = (b, h) if s_q == 1 else (b, s_q, h)
    odt = out_dtype(q.dtype)
    if out is None:
        out = torch.empty((b, s_q, h, HEAD_DIM_V), dtype=odt, device=dev)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    if (out.shape != (b, s_q, h, HEAD_DIM_V) or out.dtype != odt or out.stride(3) != 1
            or (s_q > 1 and out.stride(1) != h * out.stride(2))):
        raise ValueError(f"out must be [b, s, h, 512] in {odt}, contiguous columns, "
                         "evenly strided rows")
    if (tuple(lse.shape) != lse_shape or lse.dtype != torch.float32 or lse.stride(-1) != 1
            or (s_q > 1 and lse.stride(1) != h)):
        raise ValueError(f"lse must be fp32 {list(lse_shape)} with contiguous rows")
    need = mla_workspace_size(b, rows, parts)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)

    p = FwdParams()
    p.b, p.seqlen_q, p.h, p.h_k, p.d, p.d_v = b, s_q, h, 1, HEAD_DIM, HEAD_DIM_V
    p.is_causal = 1 if is_causal else 0
    p.dtype = _DTYPE_CODE[q.dtype]
    p.softmax_scale = float(softmax_scale)
    p.q_scale, p.kv_scale = float(q_scale), float(kv_scale)
    p.fused_combine = 1 if fused_combine else 0
    p.q, p.q_batch_stride, p.q_head_stride = q.data_ptr(), q.stride(0), q.stride(2)
    p.kv_cache = kv_cache.data_ptr()
    p.kv_page_stride, p.kv_row_stride = kv_cache.stride(0), kv_cache.stride(1)
    p.num_pages, p.page_block_size = kv_cache.shape[0], kv_cache.shape[1]
    p.block_table = block_table.data_ptr()
    p.block_table_batch_stride = block_table.stride(0)
    p.max_blocks_per_seq = block_table.shape[1]
    p.cache_seqlens = cache_seqlens.data_ptr()
    p.out, p.o_batch_stride, p.o_head_stride = out.data_ptr(), out.stride(0), out.stride(2)
    p.lse, p.lse_batch_stride = lse.data_ptr(), lse.stride(0)
    p.tile_scheduler_metadata = tile_scheduler_metadata.data_ptr()
    p.num_splits = num_splits.data_ptr()
    p.num_sm_parts = parts
    p.workspace = workspace.data_ptr()
    p.workspace_bytes = workspace.numel() * workspace.element_size()
    if q_pe is not None:
        p.q_pe, p.q_pe_batch_stride, p.q_pe_head_stride = (q_pe.data_ptr(), q_pe.stride(0),
                                                           q_pe.stride(2))
    if k_pe is not None:
        p.k_pe, p.k_pe_page_stride, p.k_pe_row_stride = (k_pe.data_ptr(), k_pe.stride(0),
                                                         k_pe.stride(1))
    keep = (q, kv_cache, block_table, cache_seqlens, tile_scheduler_metadata, num_splits,
            workspace, q_pe, k_pe)
    return DecodeCall(p, keep, out, lse)


def mla_decode_fwd_timed(*args, split_events, **kw):
    """mla_decode_fwd with (begin, end) CUDA events recorded around the split kernel."""
    return mla_decode_fwd(*args, split_events=split_events, **kw)


def mla_decode_fwd_static(q, kv_cache, block_table, cache_seqlens, softmax_scale,
                          tile_scheduler_metadata, num_splits, out=None, lse=None, q_pe=None,
                          k_pe=None, is_causal=False, q_scale=1.0, kv_scale=1.0, fused_combine=False):
    """mla_decode_fwd with the library's built-in per-device scratch
    (STATIC_WORKSPACE_BYTES) in place of a workspace tensor: the C call allocates
    nothing.  Calls on one device must not overlap on the GPU.  Returns (out, lse)."""
    no_ws = torch.empty((0,), dtype=torch.uint8, device=q.device)
    call = prepare_decode(q, kv_cache, block_table, cache_seqlens, softmax_scale,
                          tile_scheduler_metadata, num_splits, out, lse, no_ws, q_pe=q_pe,
                          k_pe=k_pe, is_causal=is_causal, q_scale=q_scale, kv_scale=kv_scale,
                          fused_combine=fused_combine)
    lib = _load()
    with torch.cuda.device(call.device):
        rc = lib.mla_decode_fwd_static(ctypes.byref(call.params), _stream(call.device))
    _check(rc, "mla_decode_fwd_static")
    return call.out, call.lse


def mla_test_forced_timeout(call):
    """Test hook: run the split kernel of a prepared DecodeCall with its load warps
    switched off, so that its first wait for K data gives up after ~1 ms.  Returns
    the C status of the launch; read the recorded error with mla_get_device_error."""
    lib = _load()
    with torch.cuda.device(call.device):
        return lib.mla_test_forced_timeout(ctypes.byref(call.params), _stream(call.device))


def mla_get_device_error(device=None):
    """Synchronise the current stream and return (status, detail) of the device error word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    detail = ctypes.c_int(0)
    with torch.cuda.device(dev):
        rc = _load().mla_get_device_error(_stream(dev), ctypes.byref(detail))
    return rc, detail.value
