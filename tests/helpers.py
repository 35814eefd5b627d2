"""Shared test helpers: golden-fixture loading, library-routine decoding of storage codes,
and a numpy scatter of dense per-token K/V into the paged layout.

The scatter is written here, independently of both the oracle and the CUDA path, from the
cache views of "paged_attn.py" (split_kv_cache):
key_cache[b, h, i // x, o, i % x] and value_cache[b, h, i, o] hold token t = (b, o).
"""
from __future__ import annotations

import ast
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name: str):
    """Parse a fixture: '#' comment lines plus one Python literal."""
    with open(os.path.join(GOLDEN, name)) as f:
        body = "\n".join(ln for ln in f.read().splitlines() if not ln.lstrip().startswith("#"))
    return ast.literal_eval(body)


def eval_expr(s: str) -> float:
    """Evaluate a fixture value: a rational ("19/7"), a power ("7 * 2**-9"), "ln2 * r",
    "inf", "-0" or "nan"."""
    s = s.strip()
    if s == "-0":
        return -0.0
    try:
        return float(s)  # plain decimals keep their sign bit ("-0.0") and "inf"/"nan"
    except ValueError:
        pass
    if s.startswith("ln2"):
        r = Fraction(s.split("*")[1].strip()) if "*" in s else Fraction(1)
        return math.log(2.0) * float(r)
    if "**" in s:
        return float(eval(s, {"__builtins__": {}}, {}))  # fixture arithmetic only
    return float(Fraction(s))


def storage_to_f64(t: torch.Tensor, storage: str) -> np.ndarray:
    """Decode stored codes with library routines (numpy float16, torch bfloat16/float8)."""
    if storage == "f16":
        return t.numpy().astype(np.float64) if t.dtype == torch.float16 else \
            t.view(torch.float16).numpy().astype(np.float64)
    if storage == "bf16":
        return t.view(torch.bfloat16).to(torch.float64).numpy()
    if storage == "fp8_e4m3":
        return t.view(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    raise ValueError(storage)


def scatter_dense_to_paged(k_dense, v_dense, tables, lens, num_blocks, bs, x, nan_value):
    """k_dense/v_dense: per sequence arrays [L_s, Hk, d] (storage dtype numpy arrays).
    Returns paged key/value caches [NB, Hk, d/x, bs, x] and [NB, Hk, d, bs] with every
    slot not written left at ``nan_value``."""
    Hk, d = k_dense[0].shape[1], k_dense[0].shape[2]
    kc = np.full((num_blocks, Hk, d // x, bs, x), nan_value, dtype=k_dense[0].dtype)
    vc = np.full((num_blocks, Hk, d, bs), nan_value, dtype=v_dense[0].dtype)
    for s, L in enumerate(lens):
        for t in range(L):
            b, o = tables[s][t // bs], t % bs
            # K: split the head dimension into (d/x, x) chunks
            kc[b, :, :, o, :] = k_dense[s][t].reshape(Hk, d // x, x)
            vc[b, :, :, o] = v_dense[s][t]
    return kc, vc


def dense_attention_f64(q, k, v, scale, slopes=None):
    """softmax(scale * q k^T + slope * t) v for one sequence in float64 numpy.
    q: [H, d]; k, v: [L, H, d] (already expanded to query heads)."""
    H, d = q.shape
    L = k.shape[0]
    s = np.einsum("hd,lhd->hl", q, k) * scale
    if slopes is not None:
        s = s + np.asarray(slopes, dtype=np.float64)[:, None] * np.arange(L)[None, :]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return np.einsum("hl,lhd->hd", e / e.sum(axis=1, keepdims=True), v), s
