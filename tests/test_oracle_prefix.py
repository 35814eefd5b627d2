"""Pins for the chunked-prefix oracle ("paged_attn.py", _forward_prefix_pytorch): checks
against things other than the oracle itself.

* a hand-worked fixture (tests/golden/prefix_hand_worked.txt) with exact rational results,
  which fixes the causal boundary (token j sees chunk keys 0..j), the unmasked context and
  the GQA head grouping;
* the dense definition written out in numpy on the un-paged sequence (keys gathered from
  the cache by index arithmetic written here), with an explicit mask;
* a special case that reduces to a library routine: no cached context is causal
  self-attention, torch's scaled_dot_product_attention(is_causal=True) in float64;
* a special case that reduces to the pinned decode oracle: one new token over c cached
  tokens is single-query decode over c + 1 tokens;
* invariances (physical block permutation; GQA equals MHA with repeated kv heads) and a
  closed form (equal keys give the running mean of the visible values).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import eval_expr, load_golden, scatter_dense_to_paged, storage_to_f64


def _ctx_kv(wl, s):
    """Context keys/values of sequence s gathered from the paged cache: token t lives in
    block_tables[s][t // bs], slot t % bs; key_cache[b, h, i // x, o, i % x]."""
    c, bs, Hk, d = int(wl.context_lens[s]), wl.block_size, wl.num_kv_heads, wl.head_size
    kc = storage_to_f64(wl.key_cache, wl.q_dtype)
    vc = storage_to_f64(wl.value_cache, wl.q_dtype)
    t = np.arange(c)
    b = wl.block_tables[s].numpy()[t // bs]
    o = t % bs
    k = kc[b, :, :, o, :].reshape(c, Hk, d)     # [c, Hk, d/x, x] -> [c, Hk, d]
    v = vc[b, :, :, o]                            # [c, Hk, d]
    return k, v


def _dense_reference(wl):
    """softmax(scale q k^T + mask) v per sequence, mask = -inf where key index > c + j."""
    H, Hk, d = wl.num_heads, wl.num_kv_heads, wl.head_size
    G = H // Hk
    q = storage_to_f64(wl.query, wl.q_dtype)
    kn = storage_to_f64(wl.key, wl.q_dtype)
    vn = storage_to_f64(wl.value, wl.q_dtype)
    qsl = wl.query_start_loc.numpy()
    out = np.zeros(q.shape)
    for s in range(wl.num_seqs):
        a, e = int(qsl[s]), int(qsl[s + 1])
        if e == a:
            continue
        c = int(wl.context_lens[s])
        kctx, vctx = _ctx_kv(wl, s)
        K = np.concatenate([kctx, kn[a:e]]).repeat(G, axis=1)   # [c + n, H, d]
        V = np.concatenate([vctx, vn[a:e]]).repeat(G, axis=1)
        sc = np.einsum("jhd,thd->hjt", q[a:e], K) * wl.scale
        j = np.arange(e - a)[:, None]
        t = np.arange(c + e - a)[None, :]
        sc = np.where(t > c + j, -np.inf, sc)
        p = np.exp(sc - sc.max(axis=2, keepdims=True))
        p /= p.sum(axis=2, keepdims=True)
        out[a:e] = np.einsum("hjt,thd->jhd", p, V)
    return out


def test_hand_worked_fixture():
    g = load_golden("prefix_hand_worked.txt")
    H, Hk, d, bs, NB = g["num_heads"], g["num_kv_heads"], g["head_size"], g["block_size"], g["num_blocks"]
    nan = np.float16(np.nan)
    kd = [np.array(x, dtype=np.float16).reshape(-1, Hk, d) for x in g["context_k"]]
    vd = [np.array(x, dtype=np.float16).reshape(-1, Hk, d) for x in g["context_v"]]
    kc, vc = scatter_dense_to_paged(kd, vd, g["block_tables"], g["context_lens"], NB, bs, 8, nan)
    out = oracle.prefix(np.array(g["q"], dtype=np.float16), np.array(g["k"], dtype=np.float16),
                        np.array(g["v"], dtype=np.float16), "f16", kc, vc, num_kv_heads=Hk,
                        block_size=bs, block_tables=np.array(g["block_tables"], dtype=np.int32),
                        query_start_loc=np.array(g["query_start_loc"], dtype=np.int32),
                        context_lens=np.array(g["context_lens"], dtype=np.int32),
                        scale=float(np.float32(eval_expr(g["scale"]))))
    want = np.array([[[eval_expr(v) for v in row] for row in tok] for tok in g["out"]])
    # scale is ln 2 rounded to float32: weights move by ~1e-8 relative
    assert np.allclose(out, want, rtol=0, atol=1e-7), np.abs(out - want).max()


@pytest.mark.parametrize("name", ["prefix_tiny", "prefix_llama_gqa"])
def test_matches_dense_masked_definition(name):
    wl = workloads.make_prefix(name, reduced=True)
    ours = oracle.prefix_workload(wl)
    ref = _dense_reference(wl)
    assert np.isfinite(ours).all()
    assert np.abs(ours - ref).max() < 1e-12


def test_ragged_and_empty_chunks_match_definition():
    wl = workloads.build_prefix(num_seqs=5, num_heads=6, num_kv_heads=3, head_size=32, block_size=8,
                                context_lens=[0, 9, 16, 0, 31], query_lens=[1, 0, 17, 8, 3],
                                q_dtype="bf16", table_width=9, seed=7)
    ours = oracle.prefix_workload(wl)
    assert np.abs(ours - _dense_reference(wl)).max() < 1e-12


def test_no_context_is_causal_sdpa():
    wl = workloads.build_prefix(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                                context_lens=[0, 0], query_lens=[33, 70], seed=8)
    ours = oracle.prefix_workload(wl)
    q = torch.from_numpy(storage_to_f64(wl.query, "f16"))
    k = torch.from_numpy(storage_to_f64(wl.key, "f16")).repeat_interleave(2, dim=1)
    v = torch.from_numpy(storage_to_f64(wl.value, "f16")).repeat_interleave(2, dim=1)
    qsl = wl.query_start_loc.tolist()
    for s in range(2):
        a, e = qsl[s], qsl[s + 1]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[a:e].transpose(0, 1), k[a:e].transpose(0, 1), v[a:e].transpose(0, 1),
            is_causal=True, scale=wl.scale).transpose(0, 1).numpy()
        assert np.abs(ours[a:e] - ref).max() < 1e-12


def test_one_new_token_is_decode():
    dw = workloads.build(num_seqs=3, num_heads=8, num_kv_heads=2, head_size=64, block_size=16,
                         seq_lens=[1, 300, 777], seed=9)
    dec = oracle.decode_workload(dw)["out"].reshape(3, 8, 64)
    # the newest token of each sequence becomes the one-token chunk; the rest is context
    kc = storage_to_f64(dw.key_cache, "f16")
    vc = storage_to_f64(dw.value_cache, "f16")
    ks, vs = [], []
    for s, L in enumerate(dw.seq_lens.tolist()):
        b, o = int(dw.block_tables[s, (L - 1) // 16]), (L - 1) % 16
        ks.append(kc[b, :, :, o, :].reshape(2, 64))
        vs.append(vc[b, :, :, o])
    out = oracle.prefix(dw.query, np.array(ks, dtype=np.float16), np.array(vs, dtype=np.float16), "f16",
                        dw.key_cache, dw.value_cache, num_kv_heads=2, block_size=16,
                        block_tables=dw.block_tables, query_start_loc=np.arange(4, dtype=np.int32),
                        context_lens=(dw.seq_lens - 1).numpy(), scale=dw.scale)
    assert np.abs(out - dec).max() < 1e-12


def test_block_permutation_invariance():
    wl = workloads.make_prefix("prefix_tiny")
    base = oracle.prefix_workload(wl)
    perm = np.random.default_rng(3).permutation(wl.num_blocks)
    kc = torch.empty_like(wl.key_cache)
    vc = torch.empty_like(wl.value_cache)
    kc[torch.from_numpy(perm)] = wl.key_cache
    vc[torch.from_numpy(perm)] = wl.value_cache
    tables = torch.from_numpy(perm[wl.block_tables.numpy()].astype(np.int32))
    moved = workloads.PrefixWorkload(**{**wl.__dict__, "key_cache": kc, "value_cache": vc,
                                        "block_tables": tables})
    assert np.array_equal(oracle.prefix_workload(moved), base)


def test_gqa_equals_mha_with_repeated_kv_heads():
    wl = workloads.build_prefix(num_seqs=2, num_heads=6, num_kv_heads=2, head_size=32, block_size=16,
                                context_lens=[20, 45], query_lens=[7, 19], seed=10)
    mha = workloads.PrefixWorkload(**{
        **wl.__dict__, "num_kv_heads": 6,
        "key_cache": wl.key_cache.repeat_interleave(3, dim=1),
        "value_cache": wl.value_cache.repeat_interleave(3, dim=1),
        "key": wl.key.repeat_interleave(3, dim=1), "value": wl.value.repeat_interleave(3, dim=1)})
    assert np.array_equal(oracle.prefix_workload(wl), oracle.prefix_workload(mha))


def test_equal_keys_give_running_mean_of_values():
    wl = workloads.build_prefix(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                                context_lens=[40, 0], query_lens=[10, 6], canaries=False, seed=11)
    kvec = torch.randn(64, generator=torch.Generator().manual_seed(1)).to(torch.float16)
    kc = wl.key_cache.clone()
    kc[:] = kvec.reshape(1, 1, 8, 1, 8)
    key = wl.key.clone()
    key[:] = kvec
    wl2 = workloads.PrefixWorkload(**{**wl.__dict__, "key_cache": kc, "key": key})
    out = oracle.prefix_workload(wl2)
    vn = storage_to_f64(wl.value, "f16")
    qsl = wl.query_start_loc.tolist()
    for s in range(2):
        a, e = qsl[s], qsl[s + 1]
        c = int(wl.context_lens[s])
        V = np.concatenate([_ctx_kv(wl, s)[1], vn[a:e]]).repeat(2, axis=1)
        mean = np.cumsum(V, axis=0) / np.arange(1, len(V) + 1)[:, None, None]
        assert np.abs(out[a:e] - mean[c:]).max() < 1e-12


def test_sampled_rows_equal_full_rows():
    wl = workloads.make_prefix("prefix_tiny")
    full = oracle.prefix_workload(wl)
    rows = np.array([[0, 0], [203, 3], [5, 1], [77, 2]], dtype=np.int32)
    part = oracle.prefix_workload(wl, rows=rows)
    assert np.array_equal(part, full[rows[:, 0], rows[:, 1]])


def test_rejects_bad_arguments():
    wl = workloads.make_prefix("prefix_tiny")
    kw = dict(num_kv_heads=2, block_size=16, block_tables=wl.block_tables,
              query_start_loc=wl.query_start_loc, scale=wl.scale)
    with pytest.raises(ValueError):  # context longer than the table covers
        oracle.prefix(wl.query, wl.key, wl.value, "f16", wl.key_cache, wl.value_cache,
                      context_lens=np.array([0, 37, 4000], dtype=np.int32), **kw)
    with pytest.raises(ValueError):  # fp8 caches have no prefix path
        oracle.prefix(wl.query, wl.key, wl.value, "fp8_e4m3", wl.key_cache, wl.value_cache,
                      context_lens=wl.context_lens, **kw)
    with pytest.raises(ValueError):  # a row outside [0, T) x [0, H)
        oracle.prefix_workload(wl, rows=np.array([[204, 0]], dtype=np.int32))
