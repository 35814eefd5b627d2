"""GPU parity: pa_v2_decode_fused (the partition combine run by the last CTA of each
(sequence, head group) inside phase 1) against the fp64 oracle.

Output, max_logits and exp_sums must match the oracle exactly as for pa_v2_decode
(tmp_output is scratch here).  Covered: every named workload (reduced size, element by
element; full size on sampled rows in the benchmark's launch configuration), both
tmp_output dtypes, CTAs that merge several partitions (with and without ALiBi), a CTA that
covers a whole sequence (single pass over many partitions), back-to-back calls that reuse one
counters array across shapes (it must be left all zero), the fallback to two kernels, and
two calls in flight on separate streams with separate counters.
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
from gpu_harness import check_decode, run_decode, sample_pairs, to_device

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(autouse=True)
def _clear_device_errors():
    pa.pa_get_device_errors(reset=True)
    yield


def _counters(wl):
    return pa.decode_counters(wl.num_seqs, wl.num_heads, wl.num_kv_heads, "cuda")


@pytest.mark.parametrize("tmp16", [False, True])
@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_reduced_workloads_match_oracle(name, tmp16):
    wl = workloads.make(name, reduced=True)
    ctr = _counters(wl)
    gpu = run_decode(wl, counters=ctr, tmp_dtype=wl.query.dtype if tmp16 else torch.float32)
    check_decode(wl, gpu, oracle.decode_workload(wl), label=f"fused {name}", check_tmp=False)
    assert torch.count_nonzero(ctr) == 0
    assert pa.pa_get_device_errors() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama_gqa_decode", "long_context_gqa", "fp8_kv", "mha_alibi_ragged",
                                  "small_batch_gqa"])
def test_full_size_workloads_sampled(name):
    wl = workloads.make(name)
    ctr = _counters(wl)
    gpu = run_decode(wl, counters=ctr)
    pairs = sample_pairs(wl, n=16 if name == "long_context_gqa" else 24)
    ref = oracle.decode_workload(wl, pairs=pairs)
    check_decode(wl, gpu, ref, pairs=pairs, label=f"fused {name}", check_tmp=False)
    out, es, ml, _ = gpu
    assert torch.isfinite(out.float()).all()
    lens = wl.seq_lens.to(torch.int64)
    for s in range(wl.num_seqs):
        Ps = int(-(-int(lens[s]) // 512))
        assert torch.all(es[s, :, Ps:] == 0) and torch.all(ml[s, :, Ps:] == -float("inf"))
    assert torch.count_nonzero(ctr) == 0
    assert pa.pa_get_device_errors() == 0


@pytest.mark.parametrize("G", [1, 6, 9, 12, 16])
def test_gqa_ratios(G):
    # above 8 query heads per kv head several CTAs (head groups) share a kv head's pages and
    # each has its own arrival counter
    wl = workloads.build(num_seqs=3, num_heads=2 * G, num_kv_heads=2, head_size=128, block_size=16,
                         seq_lens=[700, 33, 2600], seed=440 + G)
    ctr = _counters(wl)
    check_decode(wl, run_decode(wl, counters=ctr), oracle.decode_workload(wl), label=f"fused G{G}", check_tmp=False)
    assert torch.count_nonzero(ctr) == 0


def test_edge_lengths_every_block_size():
    for bs in (8, 16, 32):
        wl = workloads.build(num_seqs=13, num_heads=8, num_kv_heads=2, head_size=128, block_size=bs,
                             seq_lens=[0, 1, 2, 15, 16, 17, 511, 512, 513, 1024, 1025, 1536, 2047],
                             seed=410 + bs)
        ctr = _counters(wl)
        check_decode(wl, run_decode(wl, counters=ctr), oracle.decode_workload(wl), label=f"edge bs{bs}",
                     check_tmp=False)
        assert torch.count_nonzero(ctr) == 0


def test_back_to_back_calls_reuse_counters_across_shapes():
    # one counters array sized for the largest step serves every later call on the stream
    wls = [workloads.make("llama_gqa_decode", reduced=True), workloads.make("mha_alibi_ragged", reduced=True),
           workloads.make("long_context_gqa", reduced=True)]
    ctr = torch.zeros(max(pa.decode_num_counters(w.num_seqs, w.num_heads, w.num_kv_heads) for w in wls),
                      dtype=torch.int32, device="cuda")
    refs = [oracle.decode_workload(w) for w in wls]
    devs = [to_device(w) for w in wls]
    for rnd in range(3):
        for w, r, d in zip(wls, refs, devs):
            check_decode(w, run_decode(w, d, counters=ctr), r, label=f"round {rnd} {w.name}", check_tmp=False)
            assert torch.count_nonzero(ctr) == 0


def test_fused_equals_two_kernel_path_bitwise_statistics():
    # the statistics come from the same phase-1 arithmetic on both paths
    wl = workloads.make("fp8_kv", reduced=True)
    dev = to_device(wl)
    a = run_decode(wl, dev)
    b = run_decode(wl, dev, counters=_counters(wl))
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_fallback_to_two_kernels_leaves_counters_alone():
    # 16-bit rows of 24 heads x 256 over 196 partitions exceed what the last CTA merges:
    # the call takes the two-kernel path and never touches the counters
    wl = workloads.build(num_seqs=1, num_heads=24, num_kv_heads=4, head_size=256, block_size=16,
                         seq_lens=[100000], sigma=0.5, seed=420)
    ctr = torch.full((pa.decode_num_counters(1, 24, 4),), 7, dtype=torch.int32, device="cuda")
    gpu = run_decode(wl, counters=ctr, tmp_dtype=torch.float16)
    pairs = np.array([(0, h) for h in (0, 5, 6, 23)], dtype=np.int32)
    check_decode(wl, gpu, oracle.decode_workload(wl, pairs=pairs), pairs=pairs, label="fallback")
    assert torch.all(ctr == 7)


def _launch(wl, dev, counters, stream):
    """Enqueue one fused decode on `stream` without synchronising; returns its outputs."""
    S, H, d = wl.query.shape
    P = wl.max_num_partitions
    with torch.cuda.stream(stream):
        out = torch.full((S, H, d), float("nan"), dtype=wl.query.dtype, device="cuda")
        es = torch.full((S, H, P), float("nan"), dtype=torch.float32, device="cuda")
        ml = torch.full_like(es, float("nan"))
        tmp = torch.full((S, H, P, d), float("nan"), dtype=torch.float32, device="cuda")
        pa.pa_v2_decode(out, es, ml, tmp, dev["query"], dev["key_cache"], dev["value_cache"], wl.num_kv_heads,
                        wl.scale, dev["block_tables"], dev["seq_lens"], wl.block_size, wl.max_seq_len,
                        dev["alibi"], wl.kv_cache_dtype, wl.k_scale, wl.v_scale, counters=counters, stream=stream)
    return out, es, ml, tmp


def test_two_streams_with_their_own_counters():
    wl_a = workloads.make("llama_gqa_decode", reduced=True)
    wl_b = workloads.make("fp8_kv", reduced=True)
    ra, rb = oracle.decode_workload(wl_a), oracle.decode_workload(wl_b)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    da, db = to_device(wl_a), to_device(wl_b)
    ca, cb = _counters(wl_a), _counters(wl_b)
    torch.cuda.synchronize()
    runs = []
    for _ in range(4):  # both streams' calls in flight together, each stream's calls in order
        runs.append((_launch(wl_a, da, ca, sa), _launch(wl_b, db, cb, sb)))
    torch.cuda.synchronize()
    for ga, gb in runs:
        check_decode(wl_a, tuple(t.cpu() for t in ga), ra, label="stream a", check_tmp=False)
        check_decode(wl_b, tuple(t.cpu() for t in gb), rb, label="stream b", check_tmp=False)
    assert torch.count_nonzero(ca) == 0 and torch.count_nonzero(cb) == 0


_CHILD = r"""
import sys, torch
sys.path.insert(0, {here!r}); sys.path.insert(0, {root!r})
import oracle, workloads, paged_kv_cache_v2_gb300 as pa
from gpu_harness import check_decode, run_decode
for spec in {specs!r}:
    wl = workloads.build(**spec)
    ctr = pa.decode_counters(wl.num_seqs, wl.num_heads, wl.num_kv_heads, "cuda")
    ref = oracle.decode_workload(wl)
    check_decode(wl, run_decode(wl, counters=ctr), ref, label=f"fused {{spec}}", check_tmp=False)
    assert int(torch.count_nonzero(ctr)) == 0
    check_decode(wl, run_decode(wl), ref, label=f"two kernels {{spec}}")
print("child ok")
"""


def _run_child(px, specs, split=None):
    """Run the decode checks of `specs` in a fresh process with the partition stride forced
    to `px` (or, with `split`, the CTAs per partition forced to `split`); the library reads
    the overrides once per process."""
    env = dict(os.environ)
    if px:
        env["PA_DECODE_PX"] = str(px)
    if split:
        env["PA_DECODE_SPLIT"] = str(split)
    code = _CHILD.format(here=HERE, root=os.path.dirname(HERE), specs=specs)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


@pytest.mark.parametrize("px", [1, 2, 5])
def test_partition_strides(px):
    # PX = 1: one CTA covers each whole sequence (a single pass over all its partitions);
    # PX = 2, 5: CTAs fold several partitions, some CTAs have fewer than others or none
    _run_child(px, [dict(num_seqs=4, num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                         seq_lens=[3000, 1, 700, 2600], alibi=alibi, seed=430 + alibi) for alibi in (False, True)])


def test_ctas_merging_several_partitions_head_size_256():
    # 8 query heads of head size 256 per CTA, three to six partitions folded per CTA, both
    # query dtypes, with and without ALiBi (the merge weights are relative to the last token)
    _run_child(4, [dict(num_seqs=3, num_heads=16, num_kv_heads=2, head_size=256, block_size=16,
                        seq_lens=[9000, 4097, 11264], q_dtype=q, alibi=alibi, seed=400 + alibi)
                   for q in ("f16", "bf16") for alibi in (False, True)])


_SPLIT_SPECS = [
    dict(num_seqs=13, num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
         seq_lens=[0, 1, 2, 15, 16, 17, 511, 512, 513, 1024, 1025, 1536, 2047], seed=450),
    dict(num_seqs=3, num_heads=8, num_kv_heads=8, head_size=96, block_size=32, seq_lens=[8000, 700, 1],
         q_dtype="bf16", alibi=True, seed=451),
    dict(num_seqs=4, num_heads=12, num_kv_heads=3, head_size=128, block_size=8, seq_lens=[1030, 64, 2500, 517],
         kv_cache_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07, seed=452),
    dict(num_seqs=3, num_heads=32, num_kv_heads=2, head_size=64, block_size=16, seq_lens=[700, 33, 1500], seed=453),
    dict(num_seqs=2, num_heads=24, num_kv_heads=4, head_size=256, block_size=16, seq_lens=[3000, 2561],
         sigma=0.5, seed=454),
]


@pytest.mark.parametrize("split", [2, 4])
def test_cluster_split_partitions(split):
    # 2 or 4 CTAs of a cluster share each partition's pages; the partners' partials merge in
    # the first CTA through distributed shared memory (edge lengths, ALiBi over 8K tokens,
    # fp8 caches with block size 8, 16 query heads per kv head, head size 256)
    _run_child(None, _SPLIT_SPECS, split=split)
