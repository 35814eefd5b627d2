"""GPU parity: pa_v2_decode_append (the cache writer of each sequence's newest token fused
into phase 1) against the fp64 oracle: the oracle writer stores the new rows at the token's
slot, then the oracle decode attends over the updated caches.

Checked: the output and the partition statistics as for pa_v2_decode (tmp_output is scratch
for this entry point), and the caches after the call bit for bit (only the new tokens' slots
change).  The full-size long-context step runs CTAs that fold ten partitions each into one
row and phase 2 over those rows.  Covered: every named
workload at reduced size, edge lengths for every block size, fp8 caches with both query
dtypes, ALiBi, more than 8 query heads per kv head (several CTAs share the page; one writes
it), strided rows, a new token on a page outside the cache (masked and flagged), CTAs
striding over partitions and the cluster split.
"""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import check_decode, device_scales, sample_pairs

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(autouse=True)
def _clear_device_errors():
    pa.pa_get_device_errors(reset=True)
    yield


def _as_int(t: torch.Tensor) -> np.ndarray:
    return (t.view(torch.uint8) if t.dtype == torch.uint8 else t.view(torch.int16)).cpu().numpy()


def oracle_append(wl, slots=None):
    """The oracle caches after the writer, and the oracle decode over them."""
    kr, vr = oracle._np(wl.key_cache).copy(), oracle._np(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key, wl.new_value, wl.q_dtype, kr, vr, wl.kv_storage,
                             wl.slot_mapping if slots is None else slots, block_size=wl.block_size,
                             k_scale=wl.k_scales_or_scalar(), v_scale=wl.v_scales_or_scalar())
    return kr, vr, oracle.decode_workload(wl, key_cache=kr, value_cache=vr)


def run_append(wl, key=None, value=None, order=None):
    """pa_v2_decode_append on device copies of the workload; returns (out, es, ml, tmp), caches.
    ``order``: an int32 CUDA scratch for the grid order, or None."""
    dev = "cuda"
    S, H, d = wl.query.shape
    P = wl.max_num_partitions
    q = wl.query.to(dev)
    kc, vc = wl.key_cache.to(dev), wl.value_cache.to(dev)
    bt, sl = wl.block_tables.to(dev), wl.seq_lens.to(dev)
    slopes = None if wl.alibi_slopes is None else wl.alibi_slopes.to(dev)
    out = torch.full((S, H, d), float("nan"), dtype=wl.query.dtype, device=dev)
    es = torch.full((S, H, P), float("nan"), dtype=torch.float32, device=dev)
    ml = torch.full_like(es, float("nan"))
    tmp = torch.full((S, H, P, d), float("nan"), dtype=torch.float32, device=dev)
    nk = wl.new_key.to(dev) if key is None else key
    nv = wl.new_value.to(dev) if value is None else value
    ks, vs = device_scales(wl)
    pa.pa_v2_decode_append(out, es, ml, tmp, q, nk, nv, kc, vc, wl.num_kv_heads, wl.scale, bt, sl, wl.block_size,
                           wl.max_seq_len, slopes, wl.kv_cache_dtype, ks, vs, order=order)
    torch.cuda.synchronize()
    return (out.cpu(), es.cpu(), ml.cpu(), tmp.cpu()), kc.cpu(), vc.cpu()


def _check_all(wl, label, order=None):
    kr, vr, ref = oracle_append(wl)
    gpu, kc, vc = run_append(wl, order=order)
    # tmp_output is scratch here (CTAs streaming several partitions fold them into one row)
    check_decode(wl, gpu, ref, label=label, check_tmp=False)
    assert np.array_equal(_as_int(kc), kr.view(np.uint8 if kr.dtype == np.uint8 else np.int16)), f"{label}: key cache"
    assert np.array_equal(_as_int(vc), vr.view(np.uint8 if vr.dtype == np.uint8 else np.int16)), f"{label}: value cache"


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_reduced_workloads(name):
    _check_all(workloads.make(name, reduced=True), f"append {name}")
    assert pa.pa_get_device_errors() == 0


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_edge_lengths(bs):
    wl = workloads.build(num_seqs=13, num_heads=8, num_kv_heads=2, head_size=128, block_size=bs,
                         seq_lens=[0, 1, 2, 15, 16, 17, 511, 512, 513, 1024, 1025, 1536, 2047], seed=500 + bs)
    _check_all(wl, f"append bs{bs}")


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("kv", ["auto", "fp8_e4m3"])
@pytest.mark.parametrize("alibi", [False, True])
def test_dtypes_alibi(q_dtype, kv, alibi):
    wl = workloads.build(num_seqs=5, num_heads=12, num_kv_heads=3, head_size=128, block_size=16,
                         seq_lens=[1, 517, 1030, 64, 2500], q_dtype=q_dtype, kv_cache_dtype=kv, alibi=alibi,
                         k_scale=0.05 if kv != "auto" else 1.0, v_scale=0.07 if kv != "auto" else 1.0, seed=510)
    _check_all(wl, f"append {q_dtype} {kv} alibi={alibi}")


@pytest.mark.parametrize("G", [12, 16])
def test_more_than_eight_heads_per_kv_head(G):
    wl = workloads.build(num_seqs=3, num_heads=2 * G, num_kv_heads=2, head_size=96, block_size=32,
                         seq_lens=[700, 33, 1500], q_dtype="bf16", seed=520 + G)
    _check_all(wl, f"append G{G}")


def test_strided_rows():
    wl = workloads.make("llama_gqa_decode", reduced=True)
    S, Hk, d = wl.new_key.shape
    buf = torch.zeros(S, 3 * Hk * d, dtype=wl.new_key.dtype, device="cuda")
    buf[:, :Hk * d] = wl.new_key.reshape(S, -1).cuda()
    buf[:, 2 * Hk * d:] = wl.new_value.reshape(S, -1).cuda()
    key = buf[:, :Hk * d].view(S, Hk, d)
    value = buf[:, 2 * Hk * d:].view(S, Hk, d)
    kr, vr, ref = oracle_append(wl)
    gpu, kc, vc = run_append(wl, key, value)
    check_decode(wl, gpu, ref, label="strided rows", check_tmp=False)
    assert np.array_equal(_as_int(kc), kr.view(np.int16)) and np.array_equal(_as_int(vc), vr.view(np.int16))


def test_new_token_on_a_page_outside_the_cache_is_masked_and_flagged():
    wl = workloads.build(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                         seq_lens=[100, 40], seed=530)
    bad = wl.block_tables.clone()
    bad[0, 6] = wl.num_blocks + 3  # tokens 96..99 of sequence 0, the new token among them
    wlb = workloads.Workload(**{**wl.__dict__, "block_tables": bad})
    gpu, kc, vc = run_append(wlb)
    assert pa.pa_get_device_errors() & 1
    # nothing was written (the new token of sequence 1 is, as its page is in the cache)
    kr, vr = oracle._np(wl.key_cache).copy(), oracle._np(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key[1:], wl.new_value[1:], wl.q_dtype, kr, vr, wl.kv_storage,
                             wl.slot_mapping[1:], block_size=wl.block_size)
    assert np.array_equal(_as_int(kc), kr.view(np.int16)) and np.array_equal(_as_int(vc), vr.view(np.int16))
    # sequence 0 attends over its first 96 tokens only (no ALiBi: order does not matter)
    wl_ref = workloads.Workload(**{**wl.__dict__, "block_tables": wl.block_tables[:1].clone(),
                                   "seq_lens": torch.tensor([96], dtype=torch.int32), "num_seqs": 1,
                                   "query": wl.query[:1].clone()})
    ref0 = oracle.decode_workload(wl_ref)
    got0 = gpu[0][0].double().numpy()
    assert np.abs(got0 - ref0["out"].reshape(got0.shape)).max() <= 2e-3 + 2 ** -11 * np.abs(ref0["out"]).max()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama_gqa_decode", "long_context_gqa", "mha_alibi_ragged"])
def test_full_size_sampled(name):
    # the benchmark's launch configuration (for the long context: one wave of CTAs, each
    # folding about ten partitions into one row, and phase 2 over those rows; for the ragged
    # MHA batch: CTAs striding over partitions, sequences served longest first)
    wl = workloads.make(name)
    pairs = sample_pairs(wl, n=16)
    kr, vr = oracle._np(wl.key_cache).copy(), oracle._np(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key, wl.new_value, wl.q_dtype, kr, vr, wl.kv_storage, wl.slot_mapping,
                             block_size=wl.block_size, k_scale=wl.k_scale, v_scale=wl.v_scale)
    ref = oracle.decode_workload(wl, pairs=pairs, key_cache=kr, value_cache=vr)
    order = torch.full((wl.num_seqs,), -1, dtype=torch.int32, device="cuda")
    gpu, kc, vc = run_append(wl, order=order)
    if name == "mha_alibi_ragged":  # the grid was ordered: the scratch holds a permutation
        assert sorted(order.cpu().tolist()) == list(range(wl.num_seqs))
    check_decode(wl, gpu, ref, pairs=pairs, label=f"append {name}", check_tmp=False)
    assert np.array_equal(_as_int(kc), kr) and np.array_equal(_as_int(vc), vr)
    assert pa.pa_get_device_errors() == 0


_CHILD = r"""
import sys
sys.path.insert(0, {here!r}); sys.path.insert(0, {root!r})
import torch
import workloads
from test_parity_append import _check_all
for spec in {specs!r}:
    wl = workloads.build(**spec)
    order = torch.full((wl.num_seqs,), -1, dtype=torch.int32, device="cuda") if {order!r} else None
    _check_all(wl, f"child {{spec}}", order=order)
    if order is not None and wl.num_seqs >= 16:
        assert sorted(order.cpu().tolist()) == list(range(wl.num_seqs)), "grid order not written"
print("child ok")
"""


@pytest.mark.parametrize("env", [{"PA_DECODE_PX": "2"}, {"PA_DECODE_SPLIT": "2"}, {"PA_DECODE_SPLIT": "4"}])
def test_strides_and_cluster_split(env):
    # the CTA that streams the newest token's page is the last of its stride, or a cluster
    # partner other than the first one
    specs = [dict(num_seqs=4, num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                  seq_lens=[3000, 1, 700, 2600], alibi=True, seed=540),
             dict(num_seqs=3, num_heads=12, num_kv_heads=3, head_size=128, block_size=8, seq_lens=[1030, 64, 2500],
                  kv_cache_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07, seed=541)]
    code = _CHILD.format(here=HERE, root=os.path.dirname(HERE), specs=specs, order=False)
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


def test_grid_order_is_a_longest_first_permutation():
    rng = np.random.default_rng(560)
    lens = np.concatenate([rng.integers(0, 60000, size=997), [0, 1, 600000]]).astype(np.int32)
    sl = torch.from_numpy(lens).cuda()
    order = torch.full((lens.size,), -1, dtype=torch.int32, device="cuda")
    pa.pa_v2_decode_order(sl, order)
    torch.cuda.synchronize()
    o = order.cpu().numpy()
    assert sorted(o.tolist()) == list(range(lens.size))
    parts = np.minimum(-(-lens.astype(np.int64) // 512), 1023)[o]
    assert np.all(np.diff(parts) <= 0)


def test_strided_grid_in_longest_first_order():
    # one CTA per (sequence, kv head) streaming all its partitions, sequences served longest
    # first: same results
    specs = [dict(num_seqs=20, num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                  seq_lens=[3000, 1, 700, 2600, 0, 512, 513, 1500, 2999, 17] * 2, alibi=True, seed=570),
             dict(num_seqs=24, num_heads=12, num_kv_heads=3, head_size=128, block_size=8,
                  seq_lens=[1030, 64, 2500, 3072, 1, 777] * 4, kv_cache_dtype="fp8_e4m3", k_scale=0.05,
                  v_scale=0.07, seed=571)]
    code = _CHILD.format(here=HERE, root=os.path.dirname(HERE), specs=specs, order=True)
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, PA_DECODE_PX="1"), capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
