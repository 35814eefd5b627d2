"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on a workload and
compare it with the fp64 oracle under the stated tolerances.

Tolerances (decode): output max-abs error <= 2e-3 for fp16/bf16 caches and <= 2e-2 for an
fp8 cache, each plus half an ulp of the output dtype at the reference value (the kernel
must round its fp32 result to fp16/bf16); max_logits within 1e-4 * max(|ref|, 1);
exp_sums within relative 1e-4; unused partitions exactly -inf / 0.  Cache writes: bit-exact.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa

TOL_OUT = {"auto": 2e-3, "fp8_e4m3": 2e-2}
TOL_STAT = 1e-4


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Half the spacing of the output format at |ref| (normal range; subnormals use the
    smallest normal spacing)."""
    mant = 10 if dtype == "f16" else 7
    emin = -14 if dtype == "f16" else -126
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return 0.5 * 2.0 ** (e - mant)


def to_device(wl, device="cuda"):
    return dict(
        query=wl.query.to(device), key_cache=wl.key_cache.to(device),
        value_cache=wl.value_cache.to(device), block_tables=wl.block_tables.to(device),
        seq_lens=wl.seq_lens.to(device),
        alibi=None if wl.alibi_slopes is None else wl.alibi_slopes.to(device),
    )


def device_scales(wl):
    """The workload's k/v scales as the binding takes them: two floats, or two float32 CUDA
    tensors of num_kv_heads values (per-kv-head scales)."""
    if wl.k_scales is None:
        return wl.k_scale, wl.v_scale
    return wl.k_scales.to("cuda"), wl.v_scales.to("cuda")


def run_decode(wl, dev=None, max_num_partitions=None, max_seq_len=None, poison=True,
               tmp_dtype=torch.float32, counters=None, stream=None):
    """pa_v2_decode on a workload (pa_v2_decode_fused when `counters` is given); returns CPU
    tensors (out, exp_sums, max_logits, tmp)."""
    if dev is None:
        dev = to_device(wl)
    S, H, d = wl.query.shape
    msl = wl.max_seq_len if max_seq_len is None else max_seq_len
    P = max(1, -(-msl // 512)) if max_num_partitions is None else max_num_partitions
    fill = float("nan") if poison else 0.0
    out = torch.full((S, H, d), fill, dtype=wl.query.dtype, device="cuda")
    es = torch.full((S, H, P), fill, dtype=torch.float32, device="cuda")
    ml = torch.full((S, H, P), fill, dtype=torch.float32, device="cuda")
    tmp = torch.full((S, H, P, d), fill, dtype=tmp_dtype, device="cuda")
    ks, vs = device_scales(wl)
    pa.pa_v2_decode(out, es, ml, tmp, dev["query"], dev["key_cache"], dev["value_cache"],
                    wl.num_kv_heads, wl.scale, dev["block_tables"], dev["seq_lens"], wl.block_size,
                    msl, dev["alibi"], wl.kv_cache_dtype, ks, vs, counters=counters,
                    stream=stream)
    torch.cuda.synchronize()
    return out.cpu(), es.cpu(), ml.cpu(), tmp.cpu()


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def check_decode(wl, gpu, ref, pairs=None, label="", check_tmp=True):
    """Compare GPU results with oracle results (optionally only on (s, h) pairs).
    With a 16-bit tmp_output each partition's output is rounded once more to the output
    dtype, so both the tmp and the output bounds add half an ulp of the largest partition
    value.  check_tmp=False skips tmp_output (scratch for pa_v2_decode_fused).  Returns a
    dict of the worst errors seen."""
    out, es, ml, tmp = gpu
    tmp16 = tmp.dtype != torch.float32
    H = wl.num_heads
    P = es.shape[2]
    if pairs is None:
        pairs = ref["pairs"]
    pairs = np.asarray(pairs).reshape(-1, 2)
    lens = wl.seq_lens.numpy()
    tol = TOL_OUT[wl.kv_cache_dtype]
    worst = {"out": 0.0, "out_excess": -1.0, "ml": 0.0, "es": 0.0, "tmp": 0.0}
    for n, (s, h) in enumerate(pairs):
        L = int(lens[s])
        Ps = -(-L // 512) if L > 0 else 0
        r_out = ref["out"][n]
        g_out = out_f64(out[s, h])
        err = np.abs(g_out - r_out)
        allow = tol + half_ulp(r_out, wl.q_dtype)
        if tmp16 and Ps > 1:
            allow = allow + half_ulp(np.abs(ref["tmp_out"][n, :Ps]).max(axis=0), wl.q_dtype)
        assert np.all(np.isfinite(g_out)), f"{label} non-finite output at s={s} h={h}"
        bad = err > allow
        assert not bad.any(), (f"{label} output mismatch s={s} h={h} L={L}: max err "
                               f"{err.max():.3g} at i={int(err.argmax())} (allow {allow[err.argmax()]:.3g})")
        worst["out"] = max(worst["out"], float(err.max()))
        worst["out_excess"] = max(worst["out_excess"], float((err - tol).max()))
        for p in range(P):
            gm, ge = float(ml[s, h, p]), float(es[s, h, p])
            if p < Ps:
                rm, re_ = ref["max_logits"][n, p], ref["exp_sums"][n, p]
                dm = abs(gm - rm)
                assert dm <= TOL_STAT * max(abs(rm), 1.0), f"{label} max_logit s={s} h={h} p={p}: {gm} vs {rm}"
                de = abs(ge - re_) / re_
                assert de <= TOL_STAT, f"{label} exp_sum s={s} h={h} p={p}: {ge} vs {re_}"
                worst["ml"] = max(worst["ml"], dm / max(abs(rm), 1.0))
                worst["es"] = max(worst["es"], de)
                if Ps > 1 and check_tmp:
                    rt = ref["tmp_out"][n, p]
                    te = np.abs(tmp[s, h, p].double().numpy() - rt)
                    tallow = tol + (half_ulp(rt, wl.q_dtype) if tmp16 else 0.0)
                    assert np.all(te <= tallow), f"{label} tmp_output s={s} h={h} p={p}: err {te.max()}"
                    worst["tmp"] = max(worst["tmp"], float(te.max()))
            else:
                assert gm == -math.inf and ge == 0.0, f"{label} unused partition s={s} h={h} p={p}: {gm}, {ge}"
        if L == 0:
            assert np.all(g_out == 0.0)
    return worst


def sample_pairs(wl, n=24, seed=0):
    """A spread of (s, h) pairs: the longest and shortest sequences, every forced edge
    length, then random ones."""
    rng = np.random.default_rng(seed)
    lens = wl.seq_lens.numpy()
    S, H = wl.num_seqs, wl.num_heads
    seqs = [int(lens.argmax()), int(lens.argmin())] + [int(i) for i in np.nonzero(lens <= 1)[0][:4]]
    seqs += [int(x) for x in rng.integers(0, S, size=n)]
    pairs = []
    for i, s in enumerate(seqs[:n]):
        pairs.append((s, int(rng.integers(0, H)) if i > 1 else (0 if i == 0 else H - 1)))
    return np.array(pairs, dtype=np.int32)


# ---- chunked-prefix attention ------------------------------------------------------------
# Tolerance (prefix): output max-abs error <= 2e-3 plus half an ulp of the output dtype at
# the reference value, the decode bar for 16-bit caches.
TOL_PREFIX = 2e-3


def prefix_to_device(wl, device="cuda"):
    return {k: getattr(wl, k).to(device) for k in
            ("query", "key", "value", "key_cache", "value_cache", "block_tables", "query_start_loc",
             "context_lens")}


def run_prefix(wl, dev=None, max_query_len=None, poison=True, q_rows=None, kv_rows=None, max_splits=None,
               min_split_keys=0):
    """pa_prefix on a chunked-prefill workload; returns the CPU output [T, H, d].
    q_rows / kv_rows: optional wider row buffers the inputs are copied into (strided views);
    max_splits / min_split_keys: how contexts are cut into parts (binding defaults)."""
    if dev is None:
        dev = prefix_to_device(wl)
    q, k, v = dev["query"], dev["key"], dev["value"]
    if q_rows is not None:
        buf = torch.zeros(q.shape[0], q_rows, dtype=q.dtype, device="cuda")
        buf[:, : q.shape[1] * q.shape[2]] = q.reshape(q.shape[0], -1)
        q = buf[:, : q.shape[1] * q.shape[2]].view(q.shape[0], q.shape[1], q.shape[2])
    if kv_rows is not None:
        n = k.shape[1] * k.shape[2]
        buf = torch.zeros(k.shape[0], kv_rows, dtype=k.dtype, device="cuda")
        buf[:, :n] = k.reshape(k.shape[0], -1)
        buf[:, kv_rows // 2: kv_rows // 2 + n] = v.reshape(v.shape[0], -1)
        k = buf[:, :n].view(k.shape)
        v = buf[:, kv_rows // 2: kv_rows // 2 + n].view(v.shape)
    out = torch.full(wl.query.shape, float("nan") if poison else 0.0, dtype=wl.query.dtype, device="cuda")
    mql = wl.max_query_len if max_query_len is None else max_query_len
    pa.pa_prefix(out, q, k, v, dev["key_cache"], dev["value_cache"], dev["block_tables"],
                 dev["query_start_loc"], dev["context_lens"], mql, scale=wl.scale, max_splits=max_splits,
                 min_split_keys=min_split_keys)
    torch.cuda.synchronize()
    return out.cpu()


def check_prefix(wl, out, ref, rows=None, label=""):
    """Compare a GPU prefix output with the oracle (all rows, or (token, head) rows)."""
    if rows is None:
        g = out.double().numpy()
        r = ref
    else:
        rows = np.asarray(rows)
        g = out[rows[:, 0], rows[:, 1]].double().numpy()
        r = ref
    assert np.isfinite(g).all(), f"{label}: non-finite output"
    err = np.abs(g - r)
    allow = TOL_PREFIX + half_ulp(r, wl.q_dtype)
    bad = err > allow
    if bad.any():
        idx = np.unravel_index(int(np.argmax(err - allow)), err.shape)
        raise AssertionError(f"{label}: prefix mismatch at {idx}: err {err[idx]:.3g} allow {allow[idx]:.3g}")
    return float(err.max())


def prefix_sample_rows(wl, n=48, seed=0):
    """(token, head) rows: first and last token of every sequence's chunk, tokens around
    64-key tile edges, then random ones."""
    rng = np.random.default_rng(seed)
    qsl = wl.query_start_loc.numpy()
    H = wl.num_heads
    toks = []
    for s in range(wl.num_seqs):
        a, e = int(qsl[s]), int(qsl[s + 1])
        if e > a:
            toks += [a, e - 1] + [a + j for j in (63, 64, 127, 128) if a + j < e]
    T = int(qsl[-1])
    toks += [int(x) for x in rng.integers(0, T, size=max(0, n - len(toks)))]
    return np.array([(t, int(rng.integers(0, H))) for t in toks], dtype=np.int32)
