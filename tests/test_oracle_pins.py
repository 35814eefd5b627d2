"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test names what fixes the expected result: the dense definition of attention
(numpy and torch SDPA in float64), invariances the method must have, closed forms,
hand-worked fixtures under tests/golden/, and library decoders of the storage formats.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (dense_attention_f64, eval_expr, load_golden, scatter_dense_to_paged,
                     storage_to_f64)

NAN16 = np.float16(np.nan)


# ----------------------------------------------------------------------------------------
# format tables (P8)
# ----------------------------------------------------------------------------------------
def test_e4m3_table_matches_torch_float8():
    ours = oracle.decode_table("fp8_e4m3")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_f16_table_matches_numpy_float16():
    ours = oracle.decode_table("f16")
    ref = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_bf16_table_matches_torch_bfloat16():
    ours = oracle.decode_table("bf16")
    ref = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_format_landmarks_from_golden():
    g = load_golden("e4m3_landmarks.txt")
    tab = oracle.decode_table("fp8_e4m3")
    for code, val in g["decode"]:
        want, got = eval_expr(val), tab[int(code, 16)]
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code
    xs = np.array([eval_expr(v) for v, _ in g["encode"]], dtype=np.float32)
    codes = oracle.encode_e4m3(xs)
    for (v, c), got in zip(g["encode"], codes):
        assert got == int(c, 16), (v, hex(got), c)
    h = load_golden("half_landmarks.txt")
    for fmt in ("f16", "bf16"):
        tab = oracle.decode_table(fmt)
        for code, val in h[fmt]:
            want, got = eval_expr(val), tab[int(code, 16)]
            if math.isnan(want):
                assert math.isnan(got)
            else:
                assert got == want and math.copysign(1, got) == math.copysign(1, want), (fmt, code)


def test_e4m3_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(200_000).astype(np.float32) * 40,
                        rng.uniform(-448, 448, 50_000).astype(np.float32),
                        (rng.standard_normal(50_000) * 1e-2).astype(np.float32)])
    ours = oracle.encode_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# ----------------------------------------------------------------------------------------
# hand-worked fixtures
# ----------------------------------------------------------------------------------------
def _golden_gqa_case():
    g = load_golden("decode_hand_worked.txt")["gqa_ln2"]
    H, Hk, d, bs, NB = g["num_heads"], g["num_kv_heads"], g["head_size"], g["block_size"], g["num_blocks"]
    q = np.array(g["q"], dtype=np.float16).reshape(1, H, d)
    k = np.array(g["k"], dtype=np.float16).reshape(-1, Hk, d)
    v = np.array(g["v"], dtype=np.float16).reshape(-1, Hk, d)
    table = np.array([g["block_table"]], dtype=np.int32)
    kc, vc = scatter_dense_to_paged([k], [v], table, [g["seq_len"]], NB, bs, 8, NAN16)
    return g, q, kc, vc, table


@pytest.mark.parametrize("part", [512, 2])
def test_golden_gqa_ln2(part):
    g, q, kc, vc, table = _golden_gqa_case()
    r = oracle.decode(q, "f16", kc, vc, "f16", num_kv_heads=1, block_size=2, block_tables=table,
                      seq_lens=np.array([3], np.int32), scale=float(np.float32(math.log(2))),
                      partition_size=part)
    exp = g[f"expect_p{part}"]
    for key in ("out", "max_logits", "exp_sums") + (("tmp_out",) if "tmp_out" in exp else ()):
        want = np.vectorize(eval_expr)(np.array(exp[key], dtype=object)).astype(np.float64)
        got = r[key]
        assert np.allclose(got, want, rtol=0, atol=1e-7), (key, got, want)


@pytest.mark.parametrize("part", [512, 4])
def test_golden_alibi_geometric(part):
    g = load_golden("decode_hand_worked.txt")["alibi_geometric"]
    L, bs, d, slope = g["seq_len"], g["block_size"], g["head_size"], g["slope"]
    rng = np.random.default_rng(0)
    k = rng.standard_normal((L, 1, d)).astype(np.float16)
    v = np.zeros((L, 1, d), dtype=np.float16)
    v[:, 0, 0] = np.arange(L)
    table = np.array([g["block_table"]], dtype=np.int32)
    kc, vc = scatter_dense_to_paged([k], [v], table, [L], g["num_blocks"], bs, 8, NAN16)
    q = np.zeros((1, 1, d), dtype=np.float16)
    r = oracle.decode(q, "f16", kc, vc, "f16", num_kv_heads=1, block_size=bs, block_tables=table,
                      seq_lens=np.array([L], np.int32), scale=g["scale"],
                      alibi_slopes=np.array([slope], np.float32), partition_size=part)
    rr = math.exp(-slope)
    lsum = (1 - rr ** L) / (1 - rr)
    out0 = sum(t * rr ** (L - 1 - t) for t in range(L)) / lsum
    assert abs(r["out"][0, 0] - out0) < 1e-12
    assert np.all(r["out"][0, 1:] == 0)
    if part == 512:
        assert abs(r["max_logits"][0, 0] - slope * (L - 1)) < 1e-12
        assert abs(r["exp_sums"][0, 0] - lsum) < 1e-12
    else:
        assert abs(r["max_logits"][0, 0] - slope * 3) < 1e-12
        assert abs(r["exp_sums"][0, 0] - (1 - rr ** 4) / (1 - rr)) < 1e-12
        assert abs(r["max_logits"][0, 1] - slope * 4) < 1e-12 and r["exp_sums"][0, 1] == 1.0


# ----------------------------------------------------------------------------------------
# P1: brute force against the dense definition (numpy and torch SDPA in float64)
# ----------------------------------------------------------------------------------------
def _random_dense_case(seed, H, Hk, d, bs, lens, storage, alibi, kscale=1.0, vscale=1.0):
    rng = np.random.default_rng(seed)
    x = 16 if storage == "fp8_e4m3" else 8
    S = len(lens)
    need = [-(-L // bs) for L in lens]
    NB = sum(need) + 3
    perm = rng.permutation(NB)
    width = max(max(need), 1)
    tables = np.full((S, width), perm[-1], dtype=np.int32)
    pos = 0
    for s, n in enumerate(need):
        tables[s, :n] = perm[pos:pos + n]
        pos += n

    def draw(shape):
        a = rng.standard_normal(shape).astype(np.float32)
        if storage == "f16":
            return torch.from_numpy(a).to(torch.float16)
        if storage == "bf16":
            return torch.from_numpy(a).to(torch.bfloat16)
        return torch.from_numpy(a * 8).to(torch.float8_e4m3fn).view(torch.uint8)

    k_t = [draw((L, Hk, d)) for L in lens]
    v_t = [draw((L, Hk, d)) for L in lens]
    qs = "bf16" if storage == "bf16" else "f16"
    q_t = draw((S, H, d)) if storage != "fp8_e4m3" else \
        torch.from_numpy(rng.standard_normal((S, H, d)).astype(np.float32)).to(torch.float16)
    # storage codes as numpy for the scatter
    def codes(t):
        return t.view(torch.int16).numpy() if t.dtype in (torch.float16, torch.bfloat16) else t.numpy()
    nanc = {"f16": np.int16(0x7E00), "bf16": np.int16(0x7FC0), "fp8_e4m3": np.uint8(0x7F)}[storage]
    kc, vc = scatter_dense_to_paged([codes(t) for t in k_t], [codes(t) for t in v_t], tables,
                                    lens, NB, bs, x, nanc)
    slopes = workloads.alibi_slopes_for(H) if alibi else None
    return dict(q_t=q_t, qs=qs, k_t=k_t, v_t=v_t, kc=kc, vc=vc, tables=tables, lens=lens,
                slopes=slopes, kscale=kscale, vscale=vscale, storage=storage, H=H, Hk=Hk, d=d, bs=bs)


@pytest.mark.parametrize("storage,H,Hk,d,bs,alibi,lens", [
    ("f16", 4, 2, 64, 16, False, [37, 600, 1]),
    ("bf16", 6, 6, 96, 32, True, [5, 513, 1030]),
    ("f16", 8, 1, 80, 8, True, [700, 17]),
    ("fp8_e4m3", 8, 2, 128, 16, False, [1100, 3]),
    ("f16", 3, 3, 120, 16, False, [2049]),
])
def test_p1_brute_force_dense(storage, H, Hk, d, bs, alibi, lens):
    c = _random_dense_case(11, H, Hk, d, bs, lens, storage, alibi, kscale=0.25, vscale=0.5)
    scale = float(np.float32(1 / math.sqrt(d)))
    r = oracle.decode(c["q_t"], c["qs"], c["kc"], c["vc"], storage, num_kv_heads=Hk, block_size=bs,
                      block_tables=c["tables"], seq_lens=np.array(lens, np.int32), scale=scale,
                      alibi_slopes=c["slopes"], k_scale=0.25, v_scale=0.5)
    G = H // Hk
    qs64 = storage_to_f64(c["q_t"], c["qs"])
    for s, L in enumerate(lens):
        k = np.repeat(storage_to_f64(c["k_t"][s], storage), G, axis=1) * 0.25
        v = np.repeat(storage_to_f64(c["v_t"][s], storage), G, axis=1) * 0.5
        want, scores = dense_attention_f64(qs64[s], k, v, scale, c["slopes"])
        got = r["out"][s * H:(s + 1) * H]
        assert np.abs(got - want).max() < 1e-12
        # torch SDPA in float64 (bias passed as a float mask)
        qt = torch.from_numpy(qs64[s])[:, None, :]  # [H, 1, d]
        kt = torch.from_numpy(k).permute(1, 0, 2)
        vt = torch.from_numpy(v).permute(1, 0, 2)
        mask = None
        if c["slopes"] is not None:
            mask = (torch.from_numpy(c["slopes"].astype(np.float64))[:, None] *
                    torch.arange(L, dtype=torch.float64)[None, :])[:, None, :]
        sd = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        assert np.abs(got - sd[:, 0, :].numpy()).max() < 1e-12
        # statistics: direct per-partition max / sum over the dense scores
        for h in range(H):
            for p in range(-(-L // 512)):
                seg = scores[h, 512 * p:512 * (p + 1)]
                m = seg.max()
                assert abs(r["max_logits"][s * H + h, p] - m) <= 1e-12 * max(1, abs(m))
                assert abs(r["exp_sums"][s * H + h, p] - np.exp(seg - m).sum()) < 1e-10


# ----------------------------------------------------------------------------------------
# P2: invariance to a permutation of the physical blocks
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "fp8_kv", "mha_alibi_ragged"])
def test_p2_block_permutation_invariance(name):
    wl = workloads.make(name, reduced=True)
    base = oracle.decode_workload(wl)
    rng = np.random.default_rng(3)
    perm = torch.from_numpy(rng.permutation(wl.num_blocks))
    kc = torch.empty_like(wl.key_cache)
    vc = torch.empty_like(wl.value_cache)
    kc[perm] = wl.key_cache
    vc[perm] = wl.value_cache
    wl2 = workloads.Workload(**{**wl.__dict__, "key_cache": kc, "value_cache": vc,
                                "block_tables": perm[wl.block_tables.long()].to(torch.int32)})
    r = oracle.decode_workload(wl2)
    for key in ("out", "max_logits", "exp_sums", "tmp_out", "out_onepass"):
        assert np.array_equal(base[key], r[key]), key


# ----------------------------------------------------------------------------------------
# P3: partition-size invariance; P5: phase-2 combine equals one softmax
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "llama_gqa_decode", "long_context_gqa", "mha_alibi_ragged"])
def test_p3_p5_partition_size_invariance(name):
    wl = workloads.make(name, reduced=True)
    ref = oracle.decode_workload(wl)
    assert np.abs(ref["out"] - ref["out_onepass"]).max() < 1e-12
    for ps in (16, 64, 0):
        r = oracle.decode_workload(wl, partition_size=ps)
        assert np.abs(r["out"] - ref["out"]).max() < 1e-12
        if ps == 0:
            # one partition: its statistics are the whole-sequence max and exp-sum
            L = wl.seq_lens.numpy().repeat(wl.num_heads)
            nz = L > 0
            assert np.all(np.isfinite(r["max_logits"][nz, 0]))
            assert np.abs(r["out"][nz] - r["tmp_out"][nz, 0]).max() < 1e-12
            # global max over partitions equals the one-partition max
            g = np.where(np.isfinite(ref["max_logits"]), ref["max_logits"], -np.inf).max(axis=1)
            assert np.abs(g[nz] - r["max_logits"][nz, 0]).max() < 1e-12
            fin = np.isfinite(ref["max_logits"])
            diff = np.where(fin, ref["max_logits"] - np.where(np.isfinite(g), g, 0)[:, None], -np.inf)
            W = (np.exp(diff) * ref["exp_sums"]).sum(axis=1)
            assert np.abs(W[nz] - r["exp_sums"][nz, 0]).max() < 1e-9


def test_p5_single_partition_output_is_tmp0():
    wl = workloads.build(num_seqs=3, num_heads=8, num_kv_heads=2, head_size=64, block_size=16,
                         seq_lens=[1, 200, 512], seed=9)
    r = oracle.decode_workload(wl)
    assert np.abs(r["out"] - r["tmp_out"][:, 0, :]).max() < 1e-14
    assert np.all(r["max_logits"].shape[1] == 1)


# ----------------------------------------------------------------------------------------
# P4: closed forms
# ----------------------------------------------------------------------------------------
def test_p4_single_token_returns_scaled_v():
    wl = workloads.build(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                         seq_lens=[1, 1], kv_cache_dtype="fp8_e4m3", k_scale=0.05,
                         v_scale=0.07, seed=4)
    r = oracle.decode_workload(wl)
    vtab = storage_to_f64(wl.value_cache, "fp8_e4m3")
    ktab = storage_to_f64(wl.key_cache, "fp8_e4m3")
    q = storage_to_f64(wl.query, "f16")
    for s in range(2):
        b = int(wl.block_tables[s, 0])
        for h in range(4):
            n = s * 4 + h
            assert np.array_equal(r["out"][n], vtab[b, h // 2, :, 0] * wl.v_scale)
            assert r["exp_sums"][n, 0] == 1.0
            k = ktab[b, h // 2, :, 0, :].reshape(-1) * wl.k_scale
            s0 = wl.scale * float(q[s, h] @ k)
            assert abs(r["max_logits"][n, 0] - s0) < 1e-12 * max(1, abs(s0))


@pytest.mark.parametrize("alibi", [False, True])
def test_p4_zero_query(alibi):
    wl = workloads.build(num_seqs=3, num_heads=4, num_kv_heads=4, head_size=64, block_size=16,
                         seq_lens=[1500, 512, 7], alibi=alibi, seed=6)
    wl.query.zero_()
    r = oracle.decode_workload(wl)
    vt = storage_to_f64(wl.value_cache, "f16")
    for s, L in enumerate(wl.seq_lens.tolist()):
        bt = wl.block_tables[s].tolist()
        v = np.stack([vt[bt[t // 16], :, :, t % 16] for t in range(L)])  # [L, H, d]
        for h in range(4):
            n = s * 4 + h
            if not alibi:
                assert np.abs(r["out"][n] - v[:, h].mean(axis=0)).max() < 1e-12
            for p in range(-(-L // 512)):
                t0, t1 = 512 * p, min(512 * (p + 1), L)
                if alibi:
                    sl = float(wl.alibi_slopes[h])
                    rr = math.exp(-sl)
                    assert abs(r["max_logits"][n, p] - sl * (t1 - 1)) < 1e-9
                    assert abs(r["exp_sums"][n, p] - (1 - rr ** (t1 - t0)) / (1 - rr)) < 1e-9
                else:
                    assert r["max_logits"][n, p] == 0.0
                    assert r["exp_sums"][n, p] == float(t1 - t0)


# ----------------------------------------------------------------------------------------
# P6: GQA equals MHA over kv heads repeated G times
# ----------------------------------------------------------------------------------------
def test_p6_gqa_equals_repeated_mha():
    wl = workloads.make("long_context_gqa", reduced=True)
    G = wl.num_heads // wl.num_kv_heads
    r = oracle.decode_workload(wl)
    mha = workloads.Workload(**{**wl.__dict__,
                                "num_kv_heads": wl.num_heads,
                                "key_cache": wl.key_cache.repeat_interleave(G, dim=1).contiguous(),
                                "value_cache": wl.value_cache.repeat_interleave(G, dim=1).contiguous()})
    r2 = oracle.decode_workload(mha)
    for key in ("out", "max_logits", "exp_sums", "tmp_out"):
        assert np.array_equal(r[key], r2[key]), key


# ----------------------------------------------------------------------------------------
# P7: range invariants, canaries never reach a result, unused slots
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_p7_invariants(name):
    wl = workloads.make(name, reduced=True)
    r = oracle.decode_workload(wl)
    assert not np.isnan(r["out"]).any() and not np.isnan(r["tmp_out"]).any()
    L = wl.seq_lens.numpy().astype(np.int64).repeat(wl.num_heads)
    P = r["max_logits"].shape[1]
    for n in range(len(L)):
        np_ = -(-L[n] // 512)
        for p in range(P):
            if p < np_:
                cnt = min(512, L[n] - 512 * p)
                assert 1.0 - 1e-12 <= r["exp_sums"][n, p] <= cnt + 1e-9
                assert np.isfinite(r["max_logits"][n, p])
            else:
                assert r["max_logits"][n, p] == -np.inf and r["exp_sums"][n, p] == 0.0
        if L[n] == 0:
            assert np.all(r["out"][n] == 0)


# ----------------------------------------------------------------------------------------
# P9: writer -- bitwise for fp16/bf16, RNE-satfinite e4m3 of x / k_scale for fp8
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("storage", ["f16", "bf16", "fp8_e4m3"])
def test_p9_writer(storage):
    qd = "bf16" if storage == "bf16" else "f16"
    kvd = "fp8_e4m3" if storage == "fp8_e4m3" else "auto"
    wl = workloads.build(num_seqs=5, num_heads=8, num_kv_heads=4, head_size=128, block_size=16,
                         seq_lens=[3, 40, 0, 17, 512], q_dtype=qd, kv_cache_dtype=kvd,
                         k_scale=0.05 if kvd != "auto" else 1.0,
                         v_scale=0.03 if kvd != "auto" else 1.0, seed=12)
    kc = oracle._np(wl.key_cache).copy()
    vc = oracle._np(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key, wl.new_value, qd, kc, vc, storage, wl.slot_mapping,
                             block_size=16, k_scale=wl.k_scale, v_scale=wl.v_scale)
    x = wl.x
    k_src = oracle._np(wl.new_key)
    v_src = oracle._np(wl.new_value)
    kc0 = oracle._np(wl.key_cache)
    changed = np.zeros(kc.shape, dtype=bool)
    for s, slot in enumerate(wl.slot_mapping.tolist()):
        if slot < 0:
            continue
        b, o = slot // 16, slot % 16
        if storage == "fp8_e4m3":
            kf = storage_to_f64(wl.new_key[s], qd).astype(np.float32) / np.float32(wl.k_scale)
            vf = storage_to_f64(wl.new_value[s], qd).astype(np.float32) / np.float32(wl.v_scale)
            kw = torch.from_numpy(kf).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            vw = torch.from_numpy(vf).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        else:
            kw, vw = k_src[s], v_src[s]
        assert np.array_equal(kc[b, :, :, o, :], kw.reshape(wl.num_kv_heads, -1, x))
        assert np.array_equal(vc[b, :, :, o], vw)
        changed[b, :, :, o, :] = True
    assert np.array_equal(kc[~changed], kc0[~changed])


# ----------------------------------------------------------------------------------------
# P11: per-kv-head scales (k_scales[Hk], v_scales[Hk] in place of one k_scale / v_scale)
# ----------------------------------------------------------------------------------------
def _head_slice(wl, j):
    """The workload reduced to kv head j and its query heads, with head j's scales as the
    per-tensor k_scale / v_scale."""
    G = wl.num_heads // wl.num_kv_heads
    hs = slice(j * G, (j + 1) * G)
    return workloads.Workload(**{
        **wl.__dict__, "num_heads": G, "num_kv_heads": 1,
        "query": wl.query[:, hs].contiguous(),
        "key_cache": wl.key_cache[:, j:j + 1].contiguous(),
        "value_cache": wl.value_cache[:, j:j + 1].contiguous(),
        "alibi_slopes": None if wl.alibi_slopes is None else wl.alibi_slopes[hs].contiguous(),
        "k_scale": float(wl.k_scales[j]), "v_scale": float(wl.v_scales[j]),
        "k_scales": None, "v_scales": None})


@pytest.mark.parametrize("alibi", [False, True])
def test_p11_head_scales_split_by_kv_head(alibi):
    # attention over kv head j sees only head j's keys and values: with per-head scales the
    # result for its query heads equals the per-tensor decode of that head alone at its
    # scales (a wrong head index, or a scale taken from another head, fails this)
    wl = workloads.build(num_seqs=3, num_heads=12, num_kv_heads=3, head_size=64, block_size=16,
                         seq_lens=[700, 1, 1300], kv_cache_dtype="fp8_e4m3", alibi=alibi,
                         k_scales=[0.05, 0.11, 0.02], v_scales=[0.07, 0.013, 0.3], seed=31)
    r = oracle.decode_workload(wl)
    G = 4
    for j in range(3):
        rj = oracle.decode_workload(_head_slice(wl, j))
        rows = [s * 12 + j * G + g for s in range(3) for g in range(G)]
        for key in ("out", "max_logits", "exp_sums", "tmp_out"):
            assert np.array_equal(r[key][rows], rj[key]), (j, key)
    # and the heads really differ from a decode at one shared scale
    r1 = oracle.decode_workload(workloads.Workload(**{**wl.__dict__, "k_scales": None, "v_scales": None}))
    assert not np.allclose(r["out"], r1["out"])


def test_p11_head_scales_single_token():
    # L = 1: out = v_scales[j] * V[t0], max_logit = scale * k_scales[j] * <q, K[t0]>
    ks, vs = [0.05, 0.5], [0.25, 0.03]
    wl = workloads.build(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                         seq_lens=[1, 1], kv_cache_dtype="fp8_e4m3", k_scales=ks, v_scales=vs, seed=32)
    r = oracle.decode_workload(wl)
    vtab = storage_to_f64(wl.value_cache, "fp8_e4m3")
    ktab = storage_to_f64(wl.key_cache, "fp8_e4m3")
    q = storage_to_f64(wl.query, "f16")
    for s in range(2):
        b = int(wl.block_tables[s, 0])
        for h in range(4):
            n, j = s * 4 + h, h // 2
            assert np.array_equal(r["out"][n], vtab[b, j, :, 0] * np.float64(np.float32(vs[j])))
            k = ktab[b, j, :, 0, :].reshape(-1) * np.float64(np.float32(ks[j]))
            s0 = wl.scale * float(q[s, h] @ k)
            assert abs(r["max_logits"][n, 0] - s0) < 1e-12 * max(1, abs(s0))


def test_p11_writer_head_scales():
    # head j's rows are encoded as e4m3(x / k_scales[j]) (torch's cast of the fp32 quotient)
    ks, vs = [0.05, 0.2, 0.011, 1.5], [0.03, 0.4, 0.09, 0.007]
    wl = workloads.build(num_seqs=4, num_heads=8, num_kv_heads=4, head_size=64, block_size=16,
                         seq_lens=[3, 40, 0, 17], kv_cache_dtype="fp8_e4m3", k_scales=ks, v_scales=vs,
                         seed=33)
    kc = oracle._np(wl.key_cache).copy()
    vc = oracle._np(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key, wl.new_value, "f16", kc, vc, "fp8_e4m3", wl.slot_mapping,
                             block_size=16, k_scale=wl.k_scales, v_scale=wl.v_scales)
    for s, slot in enumerate(wl.slot_mapping.tolist()):
        if slot < 0:
            continue
        b, o = slot // 16, slot % 16
        for j in range(4):
            kf = storage_to_f64(wl.new_key[s, j], "f16").astype(np.float32) / np.float32(ks[j])
            vf = storage_to_f64(wl.new_value[s, j], "f16").astype(np.float32) / np.float32(vs[j])
            kw = torch.from_numpy(kf).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            vw = torch.from_numpy(vf).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(kc[b, j, :, o, :].reshape(-1), kw), (s, j)
            assert np.array_equal(vc[b, j, :, o], vw), (s, j)


# ----------------------------------------------------------------------------------------
# P10: seeds reproduce
# ----------------------------------------------------------------------------------------
def test_p10_seeded_generation_reproduces():
    a = workloads.make("tiny")
    b = workloads.make("tiny")
    c = workloads.make("tiny", seed=77)
    for key in ("query", "key_cache", "value_cache", "block_tables", "seq_lens", "slot_mapping"):
        ta, tb = getattr(a, key).contiguous(), getattr(b, key).contiguous()
        assert torch.equal(ta.view(torch.uint8), tb.view(torch.uint8)), key
    assert not torch.equal(a.query, c.query)
    ra, rb = oracle.decode_workload(a), oracle.decode_workload(b)
    assert np.array_equal(ra["out"], rb["out"])


# ----------------------------------------------------------------------------------------
# block moves ("paged_attn.py" copy_blocks / swap_blocks)
# ----------------------------------------------------------------------------------------
def test_copy_blocks_oracle_matches_numpy_indexing_and_hand_case():
    rng = np.random.default_rng(8)
    src = rng.integers(0, 255, size=(40, 2, 8, 16, 8), dtype=np.uint8)
    dst = rng.integers(0, 255, size=(30, 2, 8, 16, 8), dtype=np.uint8)
    m = np.stack([rng.permutation(40)[:12], rng.permutation(30)[:12]], axis=1)
    want = dst.copy()
    want[m[:, 1]] = src[m[:, 0]]
    oracle.copy_blocks(dst, src, m)
    assert np.array_equal(dst, want)
    # hand case inside one cache: block b holds the value b; (0 -> 2), (3 -> 1)
    c = np.repeat(np.arange(4, dtype=np.int32)[:, None], 5, axis=1)
    oracle.copy_blocks(c, c, np.array([[0, 2], [3, 1]]))
    assert c[:, 0].tolist() == [0, 3, 0, 3]
    with pytest.raises(ValueError):
        oracle.copy_blocks(c, c, np.array([[0, 4]]))
