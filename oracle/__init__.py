"""CPU fp64 oracle for paged single-query decode attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg use this
package; the product library never imports it and it imports nothing from the product.
The arithmetic lives in ``pa_oracle.c`` (plain loops over the paged layout, fp64); this
file builds it with gcc and marshals numpy arrays through ctypes.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` (brute-force
dense attention, torch SDPA in float64, block-permutation and partition-size invariance,
closed forms, GQA = MHA on repeated heads, the hand-worked fixtures under
``tests/golden/``, and the format tables against torch's float8/bfloat16/numpy float16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpa_oracle.so")

FMT = {"f16": 0, "bf16": 1, "f32": 2, "fp8_e4m3": 3}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.pa_oracle_decode.restype = i32
            lib.pa_oracle_decode.argtypes = [P, i32, P, P, i32, i32, i32, i32, i32, i32, P, i32, P,
                                             f32, P, f32, f32, P, P, i32, i32, P, i32, P, P, P, P, P, i32]
            lib.pa_oracle_reshape_and_cache.restype = i32
            lib.pa_oracle_reshape_and_cache.argtypes = [P, P, i32, i64, i64, P, P, i32, P, i32, i32,
                                                        i32, i32, i32, f32, f32, P, P]
            lib.pa_oracle_decode_table.restype = i32
            lib.pa_oracle_decode_table.argtypes = [i32, P]
            lib.pa_oracle_prefix.restype = i32
            lib.pa_oracle_prefix.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, i32, P, i32, P, P,
                                             f32, P, i32, P, i32]
            lib.pa_oracle_copy_blocks.restype = i32
            lib.pa_oracle_copy_blocks.argtypes = [P, P, P, i32, i64, i32, i32]
            lib.pa_oracle_encode_e4m3.restype = None
            lib.pa_oracle_encode_e4m3.argtypes = [P, i64, P]
            _lib = lib
    return _lib


def _np(t) -> np.ndarray:
    """A contiguous numpy view of a CPU tensor or array holding element codes."""
    try:
        import torch

        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype in (torch.bfloat16, torch.float16):
                t = t.view(torch.int16)
            elif t.dtype == getattr(torch, "float8_e4m3fn", None):
                t = t.view(torch.uint8)
            return t.numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(t)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _scale_arg(s, num_kv_heads: int):
    """A scale given as one float (per tensor) or as num_kv_heads floats (per kv head):
    returns (the float, or 1.0) and (None, or the float32 array)."""
    if isinstance(s, (int, float)):
        return float(s), None
    a = np.ascontiguousarray(np.asarray(_np(s) if hasattr(s, "numpy") else s, dtype=np.float32).reshape(-1))
    if a.shape != (num_kv_heads,):
        raise ValueError("per-head scales need one value per kv head")
    return 1.0, a


def decode(query, q_fmt: str, key_cache, value_cache, kv_fmt: str, *, num_kv_heads: int,
           block_size: int, block_tables, seq_lens, scale: float, alibi_slopes=None,
           k_scale=1.0, v_scale=1.0, partition_size: int = 512,
           max_num_partitions: Optional[int] = None,
           pairs: Optional[Sequence[Sequence[int]]] = None, threads: int = 0) -> dict:
    """fp64 decode attention for the requested (sequence, head) pairs (all pairs by default).

    ``k_scale`` / ``v_scale``: one float, or one per kv head (a sequence of num_kv_heads).
    Returns a dict of float64 arrays: ``out`` and ``out_onepass`` [n, d], ``max_logits`` and
    ``exp_sums`` [n, Pmax], ``tmp_out`` [n, Pmax, d] and the ``pairs`` [n, 2] used.
    """
    lib = _load()
    q = _np(query)
    kc, vc = _np(key_cache), _np(value_cache)
    bt = np.ascontiguousarray(_np(block_tables), dtype=np.int32)
    sl = np.ascontiguousarray(_np(seq_lens), dtype=np.int32)
    S, H, d = q.shape
    if max_num_partitions is None:
        mx = int(sl.max()) if sl.size else 0
        ps = partition_size if partition_size > 0 else max(mx, 1)
        max_num_partitions = max(1, -(-mx // ps))
    if pairs is None:
        pr = np.array([(s, h) for s in range(S) for h in range(H)], dtype=np.int32).reshape(-1, 2)
    else:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    n = pr.shape[0]
    P = max_num_partitions
    out = np.zeros((n, d)); out1 = np.zeros((n, d))
    ml = np.zeros((n, P)); es = np.zeros((n, P)); tmp = np.zeros((n, P, d))
    sl_f = None if alibi_slopes is None else np.ascontiguousarray(_np(alibi_slopes), dtype=np.float32)
    ks, ka = _scale_arg(k_scale, num_kv_heads)
    vs, va = _scale_arg(v_scale, num_kv_heads)
    rc = lib.pa_oracle_decode(_ptr(q), FMT[q_fmt], _ptr(kc), _ptr(vc), FMT[kv_fmt], S, H,
                              num_kv_heads, d, block_size, _ptr(bt), bt.shape[1], _ptr(sl),
                              float(scale), _ptr(sl_f), ks, vs, _ptr(ka), _ptr(va),
                              int(partition_size), P, _ptr(pr), n, _ptr(out), _ptr(out1),
                              _ptr(ml), _ptr(es), _ptr(tmp), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"out": out, "out_onepass": out1, "max_logits": ml, "exp_sums": es, "tmp_out": tmp,
            "pairs": pr}


def decode_workload(wl, pairs=None, partition_size: int = 512, threads: int = 0,
                    key_cache=None, value_cache=None) -> dict:
    """``decode`` on a workload object (see the ``workloads`` package)."""
    kv_fmt = "fp8_e4m3" if wl.kv_cache_dtype == "fp8_e4m3" else wl.q_dtype
    return decode(wl.query, wl.q_dtype,
                  wl.key_cache if key_cache is None else key_cache,
                  wl.value_cache if value_cache is None else value_cache, kv_fmt,
                  num_kv_heads=wl.num_kv_heads, block_size=wl.block_size,
                  block_tables=wl.block_tables, seq_lens=wl.seq_lens, scale=wl.scale,
                  alibi_slopes=wl.alibi_slopes, k_scale=wl.k_scales_or_scalar(),
                  v_scale=wl.v_scales_or_scalar(), partition_size=partition_size,
                  max_num_partitions=wl.max_num_partitions if partition_size == 512 else None,
                  pairs=pairs, threads=threads)


def reshape_and_cache(key, value, src_fmt: str, key_cache: np.ndarray, value_cache: np.ndarray,
                      kv_fmt: str, slot_mapping, *, block_size: int, k_scale=1.0,
                      v_scale=1.0) -> None:
    """Scatter rows key/value [T, Hk, d] into the numpy caches in place (by slot).  The scales
    are one float each, or one per kv head."""
    lib = _load()
    k, v = _np(key), _np(value)
    T, Hk, d = k.shape
    sm = np.ascontiguousarray(_np(slot_mapping), dtype=np.int64)
    assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
    ks, ka = _scale_arg(k_scale, Hk)
    vs, va = _scale_arg(v_scale, Hk)
    rc = lib.pa_oracle_reshape_and_cache(_ptr(k), _ptr(v), FMT[src_fmt], Hk * d, Hk * d,
                                         _ptr(key_cache), _ptr(value_cache), FMT[kv_fmt],
                                         _ptr(sm), T, Hk, d, block_size, key_cache.shape[0],
                                         ks, vs, _ptr(ka), _ptr(va))
    if rc != 0:
        raise ValueError("oracle writer rejected the arguments")


def decode_table(fmt: str) -> np.ndarray:
    """Every code of a storage format decoded to float64 (index = code)."""
    lib = _load()
    n = 256 if fmt == "fp8_e4m3" else 65536
    out = np.zeros(n)
    lib.pa_oracle_decode_table(FMT[fmt], _ptr(out))
    return out


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """float32 values to e4m3fn codes with the writer's rounding (RNE, satfinite)."""
    lib = _load()
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(a.shape, dtype=np.uint8)
    lib.pa_oracle_encode_e4m3(_ptr(a), a.size, _ptr(out))
    return out


def copy_blocks(dst: np.ndarray, src: np.ndarray, mapping) -> None:
    """Block moves in place: dst[d] = src[s] for each (s, d) pair of mapping, in order
    (dst and src may be the same array, as in copy-on-write inside one cache)."""
    lib = _load()
    m = np.ascontiguousarray(_np(mapping), dtype=np.int64).reshape(-1, 2)
    assert dst.flags.c_contiguous and src.flags.c_contiguous
    block_bytes = dst[0].nbytes
    assert src[0].nbytes == block_bytes
    rc = lib.pa_oracle_copy_blocks(_ptr(dst), _ptr(src), _ptr(m), m.shape[0], block_bytes, src.shape[0],
                                   dst.shape[0])
    if rc != 0:
        raise ValueError("oracle copy_blocks: id out of range")


def prefix(query, key, value, fmt: str, key_cache, value_cache, *, num_kv_heads: int, block_size: int,
           block_tables, query_start_loc, context_lens, scale: float, rows=None,
           threads: int = 0) -> np.ndarray:
    """fp64 chunked-prefix attention ("paged_attn.py" _forward_prefix_pytorch): every new token
    attends to its sequence's cached context and, causally, to the new tokens up to itself.
    query [T, H, d], key/value [T, Hk, d].  Returns out [T, H, d] float64, or [len(rows), d]
    for an optional int array of (token, head) rows."""
    lib = _load()
    q, k, v = _np(query), _np(key), _np(value)
    kc, vc = _np(key_cache), _np(value_cache)
    bt = np.ascontiguousarray(_np(block_tables), dtype=np.int32)
    qsl = np.ascontiguousarray(_np(query_start_loc), dtype=np.int32)
    cl = np.ascontiguousarray(_np(context_lens), dtype=np.int32)
    T, H, d = q.shape
    if rows is None:
        rp, nr, out = None, 0, np.zeros((T, H, d))
    else:
        rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        rp, nr, out = _ptr(rr), rr.shape[0], np.zeros((rr.shape[0], d))
    rc = lib.pa_oracle_prefix(_ptr(q), _ptr(k), _ptr(v), FMT[fmt], _ptr(kc), _ptr(vc), cl.shape[0], H,
                              num_kv_heads, d, block_size, _ptr(bt), bt.shape[1], _ptr(qsl), _ptr(cl),
                              float(scale), rp, nr, _ptr(out), int(threads))
    if rc != 0:
        raise ValueError("oracle prefix rejected the arguments")
    return out


def prefix_workload(wl, rows=None, threads: int = 0) -> np.ndarray:
    """``prefix`` on a chunked-prefill workload (all rows, or the given (token, head) rows)."""
    return prefix(wl.query, wl.key, wl.value, wl.q_dtype, wl.key_cache, wl.value_cache,
                  num_kv_heads=wl.num_kv_heads, block_size=wl.block_size,
                  block_tables=wl.block_tables, query_start_loc=wl.query_start_loc,
                  context_lens=wl.context_lens, scale=wl.scale, rows=rows, threads=threads)
