"""paged_kv_cache_v2_gb300 -- Python binding of the pa_v2 C ABI (PagedAttention V2 decode on
GB300).

Argument marshalling only: every step of the computation runs in the CUDA kernels of
``libpa_v2.so`` (built from ``csrc/``).  PyTorch supplies device memory and streams.  There
is no fallback: if the library cannot be loaded, importing the binding functions fails.

Entry points mirror ``include/pa_v2.h``:

* ``pa_v2_decode(output, exp_sums, max_logits, tmp_output, query, key_cache, value_cache,
  num_kv_heads, scale, block_tables, seq_lens, block_size, max_seq_len, alibi_slopes,
  kv_cache_dtype, k_scale, v_scale)`` -- the op signature of "paged_attention_v2_pytorch.py"
  (paged_attention_v2_pytorch) without its unused tensor-parallel / block-sparse arguments.
* ``pa_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, kv_cache_dtype,
  k_scale, v_scale)`` -- "paged_attn.py" write_to_paged_cache.
* ``pa_v2_decode(..., counters=decode_counters(S, H, Hk, device))`` -- pa_v2_decode_fused:
  the same step with the partition combine inside phase 1.
* ``pa_v2_decode_append(...)`` -- the cache writer of each sequence's newest token and the
  decode in one kernel ("paged_attn.py" forward_decode after write_to_paged_cache).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

PARTITION_SIZE = 512

PA_DT_F16, PA_DT_BF16, PA_DT_F32, PA_DT_FP8_E4M3 = 0, 1, 2, 3
PA_KV_AUTO, PA_KV_FP8_E4M3 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported combination", 3: "CUDA error",
          4: "step needs more than the fixed no-allocation scratch"}
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} returned {status} ({STATUS.get(status, 'unknown')})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpa_v2.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path}")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_uint32
    lib.pa_v2_decode.restype = i32
    lib.pa_v2_decode.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, f32, P, i32, i32, P, i32, i32,
                                 i32, P, i32, i32, i32, f32, f32, P]
    lib.pa_v2_decode_fused.restype = i32
    lib.pa_v2_decode_fused.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, f32, P, i32, i32, P, i32, i32,
                                       i32, P, i32, i32, i32, f32, f32, P, i64, P]
    lib.pa_v2_decode_append.restype = i32
    lib.pa_v2_decode_append.argtypes = [P, P, P, P, P, P, P, i64, i64, P, P, i32, i32, i32, i32, f32, P, i32, i32, P,
                                        i32, i32, i32, P, i32, i32, i32, f32, f32, P, P]
    lib.pa_v2_decode_order.restype = i32
    lib.pa_v2_decode_order.argtypes = [P, i32, P, P]
    lib.pa_v2_decode_num_counters.restype = i64
    lib.pa_v2_decode_num_counters.argtypes = [i32, i32, i32]
    lib.pa_reshape_and_cache.restype = i32
    lib.pa_reshape_and_cache.argtypes = [P, P, i64, i64, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                         f32, f32, P]
    lib.pa_v2_decode_head_scales.restype = i32
    lib.pa_v2_decode_head_scales.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, f32, P, i32, i32, P, i32,
                                             i32, i32, P, i32, i32, i32, P, P, P]
    lib.pa_v2_decode_append_head_scales.restype = i32
    lib.pa_v2_decode_append_head_scales.argtypes = [P, P, P, P, P, P, P, i64, i64, P, P, i32, i32, i32, i32, f32, P,
                                                    i32, i32, P, i32, i32, i32, P, i32, i32, i32, P, P, P, P]
    lib.pa_reshape_and_cache_head_scales.restype = i32
    lib.pa_reshape_and_cache_head_scales.argtypes = [P, P, i64, i64, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                     P, P, P]
    lib.pa_v2_partition_size.restype = i32
    lib.pa_v2_partition_size.argtypes = []
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [i32]
    lib.pa_get_device_errors.restype = i32
    lib.pa_get_device_errors.argtypes = [ctypes.POINTER(u32), i32]
    lib.pa_v2_set_timing_events.restype = i32
    lib.pa_v2_set_timing_events.argtypes = [P, P]
    lib.pa_copy_blocks.restype = i32
    lib.pa_copy_blocks.argtypes = [P, P, i32, P, i32, i64, i32, P]
    lib.pa_swap_blocks.restype = i32
    lib.pa_swap_blocks.argtypes = [P, P, P, i32, i64, i32, i32, P]
    lib.pa_prefix.restype = i32
    lib.pa_prefix.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, f32, P, i32, i32, P, P, i32, i32, i64, i64,
                              i32, P, ctypes.c_size_t, i32, i32, P]
    lib.pa_prefix_workspace_size.restype = ctypes.c_size_t
    lib.pa_prefix_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pa_prefix_num_parts.restype = i32
    lib.pa_prefix_num_parts.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32)]
    lib.pa_v2_decode_noalloc.restype = i32
    lib.pa_v2_decode_noalloc.argtypes = [P, P, P, P, i32, i32, i32, i32, f32, P, i32, i32, P, i32, i32,
                                         P, i32, i32, f32, f32, P]
    _lib = lib
    return lib


def _dt(t: torch.dtype) -> int:
    if t == torch.float16:
        return PA_DT_F16
    if t == torch.bfloat16:
        return PA_DT_BF16
    raise TypeError(f"unsupported query dtype {t}")


def _kv(kv_cache_dtype: str) -> int:
    if kv_cache_dtype in ("auto", None):
        return PA_KV_AUTO
    if kv_cache_dtype in ("fp8", "fp8_e4m3"):
        return PA_KV_FP8_E4M3
    raise ValueError(f"unsupported kv_cache_dtype {kv_cache_dtype!r}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(call: str, st: int) -> None:
    if st != 0:
        raise PagedAttentionError(call, st)


def _head_scales(k_scale, v_scale, num_kv_heads: int):
    """None for per-tensor scales (two floats); the two pointers for per-kv-head scales
    (two float32 CUDA tensors of num_kv_heads values)."""
    kt, vt = isinstance(k_scale, torch.Tensor), isinstance(v_scale, torch.Tensor)
    if not kt and not vt:
        return None
    if not (kt and vt):
        raise TypeError("k_scale and v_scale must both be floats or both be per-kv-head tensors")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.numel() != num_kv_heads:
            raise TypeError(f"{name} per kv head must be a contiguous float32 CUDA tensor of num_kv_heads values")
    return _ptr(k_scale), _ptr(v_scale)


def pa_v2_decode(output: torch.Tensor, exp_sums: torch.Tensor, max_logits: torch.Tensor,
                 tmp_output: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                 value_cache: torch.Tensor, num_kv_heads: int, scale: float,
                 block_tables: torch.Tensor, seq_lens: torch.Tensor, block_size: int,
                 max_seq_len: int, alibi_slopes: Optional[torch.Tensor] = None,
                 kv_cache_dtype: str = "auto", k_scale=1.0, v_scale=1.0,
                 num_blocks: Optional[int] = None, stream=None, counters: Optional[torch.Tensor] = None) -> None:
    """Enqueue one decode step (phase 1 + phase 2) on ``stream`` (default: current stream).

    Shapes: query/output [S, H, d]; key_cache [NB, Hk, d/x, bs, x]; value_cache
    [NB, Hk, d, bs]; block_tables int32 [S, W]; seq_lens int32 [S]; exp_sums/max_logits
    fp32 [S, H, P]; tmp_output fp32 [S, H, P, d].  The fp8 cache may be passed as uint8
    codes or as torch.float8_e4m3fn.

    With ``counters`` (from :func:`decode_counters`, zeroed once when allocated) the call is
    ``pa_v2_decode_fused``: the partition combine runs inside phase 1 and tmp_output is
    scratch.  ``k_scale`` / ``v_scale`` as float32 CUDA tensors of num_kv_heads values make
    the call ``pa_v2_decode_head_scales`` (one scale per kv head).
    """
    lib = load()
    for name, t in (("output", output), ("exp_sums", exp_sums), ("max_logits", max_logits),
                    ("tmp_output", tmp_output), ("query", query), ("key_cache", key_cache),
                    ("value_cache", value_cache), ("block_tables", block_tables),
                    ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    if exp_sums.dtype != torch.float32 or max_logits.dtype != torch.float32:
        raise TypeError("exp_sums and max_logits must be float32")
    if tmp_output.dtype == torch.float32:
        tmp_dtype = PA_DT_F32
    elif tmp_output.dtype == query.dtype:
        tmp_dtype = _dt(query.dtype)
    else:
        raise TypeError("tmp_output must be float32 or the query dtype")
    if output.dtype != query.dtype:
        raise TypeError("output must have the query dtype")
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_cuda):
        raise TypeError("alibi_slopes must be a float32 CUDA tensor")
    S, H, d = query.shape
    if num_blocks is None:
        num_blocks = key_cache.shape[0]
    hs = _head_scales(k_scale, v_scale, int(num_kv_heads))
    args = (_ptr(output), _ptr(exp_sums), _ptr(max_logits), _ptr(tmp_output),
            _ptr(query), _ptr(key_cache), _ptr(value_cache), S, H, int(num_kv_heads),
            d, float(scale), _ptr(block_tables), int(block_tables.shape[1]),
            int(num_blocks), _ptr(seq_lens), int(block_size), int(max_seq_len),
            int(tmp_output.shape[2]), _ptr(alibi_slopes), _dt(query.dtype),
            _kv(kv_cache_dtype), tmp_dtype)
    if hs is not None:
        if counters is not None:
            raise TypeError("the fused combine takes per-tensor scales only")
        _check("pa_v2_decode_head_scales", lib.pa_v2_decode_head_scales(*args, *hs, _stream(stream)))
        return
    args = args + (float(k_scale), float(v_scale))
    if counters is None:
        _check("pa_v2_decode", lib.pa_v2_decode(*args, _stream(stream)))
        return
    if counters.dtype != torch.int32 or not counters.is_cuda or not counters.is_contiguous():
        raise TypeError("counters must be a contiguous int32 CUDA tensor (see decode_counters)")
    _check("pa_v2_decode_fused", lib.pa_v2_decode_fused(*args, _ptr(counters), counters.numel(), _stream(stream)))


def pa_v2_decode_append(output: torch.Tensor, exp_sums: torch.Tensor, max_logits: torch.Tensor,
                        tmp_output: torch.Tensor, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                        key_cache: torch.Tensor, value_cache: torch.Tensor, num_kv_heads: int, scale: float,
                        block_tables: torch.Tensor, seq_lens: torch.Tensor, block_size: int, max_seq_len: int,
                        alibi_slopes: Optional[torch.Tensor] = None, kv_cache_dtype: str = "auto",
                        k_scale=1.0, v_scale=1.0, num_blocks: Optional[int] = None,
                        stream=None, order: Optional[torch.Tensor] = None) -> None:
    """One decode step that first appends every sequence's newest token (key/value [S, Hk, d]
    rows, position seq_lens[s] - 1, slot from the block table) to the caches: the cache
    writer and pa_v2_decode in one kernel.  Other arguments as pa_v2_decode (per-kv-head
    scale tensors make the call ``pa_v2_decode_append_head_scales``).  ``order``: an int32
    CUDA tensor of num_seqs entries the call may use as scratch for a longest-first grid
    order (see :func:`pa_v2_decode_order`), or None."""
    lib = load()
    for name, t in (("output", output), ("exp_sums", exp_sums), ("max_logits", max_logits),
                    ("tmp_output", tmp_output), ("query", query), ("key_cache", key_cache),
                    ("value_cache", value_cache), ("block_tables", block_tables), ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    S, H, d = query.shape
    for name, t in (("key", key), ("value", value)):
        if t.dim() != 3 or t.shape[0] != S or t.shape[1] != num_kv_heads or t.shape[2] != d or \
                t.stride(2) != 1 or t.stride(1) != d or t.dtype != query.dtype or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor [num_seqs, num_kv_heads, head_size] in the query "
                             "dtype with dense rows")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    if exp_sums.dtype != torch.float32 or max_logits.dtype != torch.float32:
        raise TypeError("exp_sums and max_logits must be float32")
    if tmp_output.dtype == torch.float32:
        tmp_dtype = PA_DT_F32
    elif tmp_output.dtype == query.dtype:
        tmp_dtype = _dt(query.dtype)
    else:
        raise TypeError("tmp_output must be float32 or the query dtype")
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_cuda):
        raise TypeError("alibi_slopes must be a float32 CUDA tensor")
    if num_blocks is None:
        num_blocks = key_cache.shape[0]
    args = (_ptr(output), _ptr(exp_sums), _ptr(max_logits), _ptr(tmp_output), _ptr(query), _ptr(key), _ptr(value),
            key.stride(0), value.stride(0), _ptr(key_cache), _ptr(value_cache), S, H, int(num_kv_heads), d,
            float(scale), _ptr(block_tables), int(block_tables.shape[1]), int(num_blocks), _ptr(seq_lens),
            int(block_size), int(max_seq_len), int(tmp_output.shape[2]), _ptr(alibi_slopes), _dt(query.dtype),
            _kv(kv_cache_dtype), tmp_dtype)
    if order is not None and (order.dtype != torch.int32 or not order.is_cuda or not order.is_contiguous()
                              or order.numel() < S):
        raise TypeError("order must be a contiguous int32 CUDA tensor of num_seqs entries")
    hs = _head_scales(k_scale, v_scale, int(num_kv_heads))
    if hs is not None:
        _check("pa_v2_decode_append_head_scales",
               lib.pa_v2_decode_append_head_scales(*args, *hs, _ptr(order), _stream(stream)))
        return
    _check("pa_v2_decode_append", lib.pa_v2_decode_append(*args, float(k_scale), float(v_scale), _ptr(order),
                                                          _stream(stream)))


def pa_v2_decode_order(seq_lens: torch.Tensor, order: torch.Tensor, stream=None) -> None:
    """Write into ``order`` (int32 CUDA [num_seqs]) the sequences by decreasing partition count."""
    lib = load()
    for name, t in (("seq_lens", seq_lens), ("order", order)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    if order.numel() < seq_lens.numel():
        raise ValueError("order needs one entry per sequence")
    _check("pa_v2_decode_order", lib.pa_v2_decode_order(_ptr(seq_lens), seq_lens.numel(), _ptr(order),
                                                        _stream(stream)))


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                         kv_cache_dtype: str = "auto", k_scale=1.0, v_scale=1.0,
                         stream=None) -> None:
    """Enqueue the slot-mapping cache writer: key/value [T, Hk, d] rows into the caches
    (per-kv-head scale tensors make the call ``pa_reshape_and_cache_head_scales``)."""
    lib = load()
    if key.dim() != 3 or value.shape != key.shape:
        raise ValueError("key and value must be [num_tokens, num_kv_heads, head_size]")
    T, Hk, d = key.shape
    if key.stride(2) != 1 or key.stride(1) != d or value.stride(2) != 1 or value.stride(1) != d:
        raise ValueError("key/value rows must be contiguous [num_kv_heads, head_size]")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous():
        raise TypeError("slot_mapping must be a contiguous int64 tensor")
    bs = value_cache.shape[-1]
    args = (_ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(key_cache), _ptr(value_cache),
            _ptr(slot_mapping), T, Hk, d, int(bs), int(key_cache.shape[0]), _dt(key.dtype), _kv(kv_cache_dtype))
    hs = _head_scales(k_scale, v_scale, Hk)
    if hs is not None:
        _check("pa_reshape_and_cache_head_scales", lib.pa_reshape_and_cache_head_scales(*args, *hs, _stream(stream)))
        return
    _check("pa_reshape_and_cache", lib.pa_reshape_and_cache(*args, float(k_scale), float(v_scale), _stream(stream)))


def pa_v2_decode_head_scales(output, exp_sums, max_logits, tmp_output, query, key_cache, value_cache,
                             num_kv_heads: int, scale: float, block_tables, seq_lens, block_size: int,
                             max_seq_len: int, alibi_slopes=None, kv_cache_dtype: str = "auto", *,
                             k_scales: torch.Tensor, v_scales: torch.Tensor, num_blocks: Optional[int] = None,
                             stream=None) -> None:
    """pa_v2_decode with one k_scale / v_scale per kv head (float32 CUDA tensors [Hk])."""
    pa_v2_decode(output, exp_sums, max_logits, tmp_output, query, key_cache, value_cache, num_kv_heads, scale,
                 block_tables, seq_lens, block_size, max_seq_len, alibi_slopes, kv_cache_dtype, k_scales, v_scales,
                 num_blocks=num_blocks, stream=stream)


def pa_v2_decode_append_head_scales(output, exp_sums, max_logits, tmp_output, query, key, value, key_cache,
                                    value_cache, num_kv_heads: int, scale: float, block_tables, seq_lens,
                                    block_size: int, max_seq_len: int, alibi_slopes=None,
                                    kv_cache_dtype: str = "auto", *, k_scales: torch.Tensor,
                                    v_scales: torch.Tensor, num_blocks: Optional[int] = None, stream=None,
                                    order: Optional[torch.Tensor] = None) -> None:
    """pa_v2_decode_append with one k_scale / v_scale per kv head (float32 CUDA tensors [Hk])."""
    pa_v2_decode_append(output, exp_sums, max_logits, tmp_output, query, key, value, key_cache, value_cache,
                        num_kv_heads, scale, block_tables, seq_lens, block_size, max_seq_len, alibi_slopes,
                        kv_cache_dtype, k_scales, v_scales, num_blocks=num_blocks, stream=stream, order=order)


def pa_reshape_and_cache_head_scales(key, value, key_cache, value_cache, slot_mapping,
                                     kv_cache_dtype: str = "auto", *, k_scales: torch.Tensor,
                                     v_scales: torch.Tensor, stream=None) -> None:
    """pa_reshape_and_cache with one k_scale / v_scale per kv head (float32 CUDA tensors [Hk])."""
    pa_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, kv_cache_dtype, k_scales, v_scales,
                         stream=stream)


def pa_v2_decode_noalloc(output: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, num_kv_heads: int, scale: float,
                         block_tables: torch.Tensor, seq_lens: torch.Tensor, block_size: int,
                         max_seq_len: int, alibi_slopes: Optional[torch.Tensor] = None,
                         kv_cache_dtype: str = "auto", k_scale: float = 1.0, v_scale: float = 1.0,
                         num_blocks: Optional[int] = None, stream=None) -> None:
    """pa_v2_decode without a caller-provided workspace: for callers that cannot allocate
    device memory (a plugin handed a stream and a device-memory budget fixed at start-up).
    The workspace is the library's fixed per-device scratch, shared by every call: order the
    calls on one stream (calls that can overlap on the GPU race on it).  The call runs with
    the query's device current, since the scratch address is looked up per device."""
    lib = load()
    for name, t in (("output", output), ("query", query), ("key_cache", key_cache),
                    ("value_cache", value_cache), ("block_tables", block_tables), ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    if output.dtype != query.dtype:
        raise TypeError("output must have the query dtype")
    S, H, d = query.shape
    if num_blocks is None:
        num_blocks = key_cache.shape[0]
    with torch.cuda.device(query.device):
        st = lib.pa_v2_decode_noalloc(_ptr(output), _ptr(query), _ptr(key_cache), _ptr(value_cache), S, H,
                                      int(num_kv_heads), d, float(scale), _ptr(block_tables),
                                      int(block_tables.shape[1]), int(num_blocks), _ptr(seq_lens),
                                      int(block_size), int(max_seq_len), _ptr(alibi_slopes),
                                      _dt(query.dtype), _kv(kv_cache_dtype), float(k_scale), float(v_scale),
                                      _stream(stream))
    _check("pa_v2_decode_noalloc", st)


def pa_copy_blocks(key_caches, value_caches, block_mapping: torch.Tensor, stream=None) -> None:
    """Copy blocks inside each layer's caches ("paged_attn.py" copy_blocks): for every pair
    (src, dst) of block_mapping (int64 [n, 2], on the GPU), cache[dst] = cache[src] in every
    K and V cache of the lists.  No dst may be another pair's src."""
    lib = load()
    key_caches, value_caches = list(key_caches), list(value_caches)
    if len(key_caches) != len(value_caches) or not key_caches:
        raise ValueError("need one value cache per key cache")
    nb = key_caches[0].shape[0]
    block_bytes = key_caches[0][0].numel() * key_caches[0].element_size()
    for t in key_caches + value_caches:
        if not t.is_cuda or not t.is_contiguous() or t.shape[0] != nb or \
                t[0].numel() * t.element_size() != block_bytes:
            raise ValueError("caches must be contiguous CUDA tensors with equal block shapes")
    m = block_mapping
    if m.dtype != torch.int64 or not m.is_cuda or not m.is_contiguous() or m.dim() != 2 or m.shape[1] != 2:
        raise TypeError("block_mapping must be a contiguous int64 CUDA tensor [n, 2]")
    L = len(key_caches)
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in key_caches])
    vp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in value_caches])
    _check("pa_copy_blocks", lib.pa_copy_blocks(kp, vp, L, _ptr(m), m.shape[0], block_bytes, nb,
                                                _stream(stream)))


def pa_swap_blocks(src: torch.Tensor, dst: torch.Tensor, block_mapping: torch.Tensor, stream=None) -> None:
    """Move blocks between two caches ("paged_attn.py" swap_blocks), e.g. GPU and pinned host:
    dst[d] = src[s] for every pair (s, d) of block_mapping (int64 [n, 2], on the host)."""
    lib = load()
    if not src.is_contiguous() or not dst.is_contiguous():
        raise ValueError("caches must be contiguous")
    block_bytes = src[0].numel() * src.element_size()
    if dst[0].numel() * dst.element_size() != block_bytes:
        raise ValueError("blocks of src and dst differ in size")
    m = block_mapping
    if m.dtype != torch.int64 or m.is_cuda or m.dim() != 2 or m.shape[1] != 2:
        raise TypeError("block_mapping must be an int64 CPU tensor [n, 2]")
    m = m.contiguous()
    if stream is None:
        stream = torch.cuda.current_stream(dst.device if dst.is_cuda else src.device)
    _check("pa_swap_blocks", lib.pa_swap_blocks(_ptr(src), _ptr(dst), _ptr(m), m.shape[0], block_bytes,
                                                src.shape[0], dst.shape[0], _stream(stream)))


def pa_prefix(output: torch.Tensor, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
              key_cache: torch.Tensor, value_cache: torch.Tensor, block_tables: torch.Tensor,
              query_start_loc: torch.Tensor, context_lens: torch.Tensor, max_query_len: int,
              scale: Optional[float] = None, stream=None, workspace: Optional[torch.Tensor] = None,
              max_splits: Optional[int] = None, min_split_keys: int = 0) -> None:
    """Chunked-prefix attention ("paged_attn.py" forward_prefix): every new token attends to
    its sequence's cached context and, causally, to the chunk's tokens up to itself.
    output/query [T, H, d], key/value [T, Hk, d] (rows may be strided, last two dims dense),
    caches in the decode layouts, int32 block_tables [S, W], query_start_loc [S+1],
    context_lens [S].  scale defaults to d^-0.5 as on the pages.

    Contexts longer than min_split_keys are cut into up to max_splits parts that run on
    separate CTAs and are merged by a second kernel; min_split_keys=0 takes the library's plan
    (contexts over 16384 tokens, cut only where one sequence's CTAs would occupy fewer than
    half the SMs; prefix_num_parts says what a call will do).  workspace is a uint8 CUDA tensor
    of at least prefix_workspace_size(...) bytes; when it is None and the call would cut a
    context, one is taken from torch's allocator (max_splits defaults to 8; max_splits=1
    turns splitting off)."""
    lib = load()
    T, H, d = query.shape
    Hk = key_cache.shape[1]
    bs = value_cache.shape[3]
    for name, t in (("query", query), ("key", key), ("value", value)):
        if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != d or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor [T, heads, d] with dense heads")
    if key.stride(0) != value.stride(0):
        raise ValueError("key and value must share a row stride")
    if not output.is_contiguous() or output.shape != query.shape or output.dtype != query.dtype:
        raise ValueError("output must be a contiguous tensor shaped like query")
    for name, t in (("key_cache", key_cache), ("value_cache", value_cache)):
        if not t.is_contiguous() or t.dtype != query.dtype:
            raise ValueError(f"{name} must be contiguous in the query dtype")
    for name, t in (("block_tables", block_tables), ("query_start_loc", query_start_loc),
                    ("context_lens", context_lens)):
        if t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda:
            raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    S = context_lens.shape[0]
    if scale is None:
        scale = d ** -0.5
    if max_splits is None:
        max_splits = 8
    split_keys = min_split_keys or PREFIX_SPLIT_KEYS
    if workspace is None and max_splits > 1 and block_tables.shape[1] * bs > split_keys and prefix_num_parts(
            H, Hk, d, query.dtype, int(max_query_len), block_tables.shape[1], bs, min(max_splits, 32),
            int(min_split_keys)) > 1:
        max_splits = min(max_splits, -(-block_tables.shape[1] * bs // split_keys))
        nbytes = prefix_workspace_size(S, H, Hk, d, int(max_query_len), max_splits)
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=query.device)
            if stream is not None:
                workspace.record_stream(stream)  # not reused before the call's work on `stream` ends
    if workspace is not None and (workspace.dtype != torch.uint8 or not workspace.is_cuda
                                  or not workspace.is_contiguous()):
        raise TypeError("workspace must be a contiguous uint8 CUDA tensor")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel())
    _check("pa_prefix", lib.pa_prefix(
        _ptr(output), _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), S, H, Hk, d,
        float(scale), _ptr(block_tables), block_tables.shape[1], key_cache.shape[0], _ptr(query_start_loc),
        _ptr(context_lens), int(max_query_len), bs, query.stride(0), key.stride(0), _dt(query.dtype),
        ws_ptr, ws_bytes, int(max_splits), int(min_split_keys), _stream(stream)))


# Default shortest context (tokens) that pa_prefix cuts into parts.
PREFIX_SPLIT_KEYS = 16384


def prefix_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_size: int,
                          max_query_len: int, max_splits: int) -> int:
    """Bytes of workspace pa_prefix needs to cut contexts into up to max_splits parts."""
    return int(load().pa_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_query_len,
                                               max_splits))


def prefix_num_parts(num_heads: int, num_kv_heads: int, head_size: int, dtype: torch.dtype, max_query_len: int,
                     max_blocks_per_seq: int, block_size: int, max_splits: int = 8, min_split_keys: int = 0,
                     has_workspace: bool = True) -> int:
    """Parts each context is cut into by a pa_prefix call with these arguments (1: no cut)."""
    out = ctypes.c_int(0)
    _check("pa_prefix_num_parts", load().pa_prefix_num_parts(
        num_heads, num_kv_heads, head_size, _dt(dtype), max_query_len, max_blocks_per_seq, block_size, max_splits,
        min_split_keys, 1 if has_workspace else 0, ctypes.byref(out)))
    return int(out.value)


def pa_v2_partition_size() -> int:
    return int(load().pa_v2_partition_size())


def pa_status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def pa_get_device_errors(reset: bool = True) -> int:
    """Device-side error flags of the current device (synchronises the device)."""
    v = ctypes.c_uint32(0)
    _check("pa_get_device_errors", load().pa_get_device_errors(ctypes.byref(v), 1 if reset else 0))
    return int(v.value)


def pa_v2_set_timing_events(begin: Optional[torch.cuda.Event], end: Optional[torch.cuda.Event]) -> None:
    """Record ``begin``/``end`` around every later phase-1 launch (None, None to stop)."""
    b = None if begin is None else ctypes.c_void_p(begin.cuda_event)
    e = None if end is None else ctypes.c_void_p(end.cuda_event)
    _check("pa_v2_set_timing_events", load().pa_v2_set_timing_events(b, e))


def decode_num_counters(num_seqs: int, num_heads: int, num_kv_heads: int) -> int:
    """Arrival counters pa_v2_decode_fused needs for a step of this shape."""
    return int(load().pa_v2_decode_num_counters(num_seqs, num_heads, num_kv_heads))


def decode_counters(num_seqs: int, num_heads: int, num_kv_heads: int, device) -> torch.Tensor:
    """Zeroed arrival counters for pa_v2_decode_fused (int32 storage of the uint32 array).
    Every fused call leaves them at zero, so one array serves every later call on one
    stream; calls that can overlap need one array each."""
    return torch.zeros(max(1, decode_num_counters(num_seqs, num_heads, num_kv_heads)), dtype=torch.int32,
                       device=device)


def workspace(num_seqs: int, num_heads: int, head_size: int, max_seq_len: int, device,
              tmp_dtype: torch.dtype = torch.float32) -> tuple:
    """Allocate (exp_sums, max_logits, tmp_output) for a decode step (caller-owned);
    tmp_dtype may be float32 or the query dtype."""
    P = max(1, -(-max_seq_len // PARTITION_SIZE))
    es = torch.empty((num_seqs, num_heads, P), dtype=torch.float32, device=device)
    ml = torch.empty_like(es)
    tmp = torch.empty((num_seqs, num_heads, P, head_size), dtype=tmp_dtype, device=device)
    return es, ml, tmp
