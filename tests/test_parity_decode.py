"""GPU parity: pa_v2_decode (through the C ABI) against the fp64 oracle on the same seeded
inputs.  Reduced-size versions of the five decode workloads are compared element by
element; the full-size workloads (in the launch configuration the benchmark times) are
compared on a sample of (sequence, head) rows.  Edge cases: empty and one-token sequences,
partition boundaries, every supported head size and block size, GQA ratios 1..16, ALiBi,
fp8 caches with both query dtypes, extra unused partitions, NaN canaries everywhere a
masked slot could leak from, and out-of-range table entries (masked and flagged)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import check_decode, run_decode, sample_pairs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_errors():
    pa.pa_get_device_errors(reset=True)
    yield


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_reduced_workloads_match_oracle(name):
    wl = workloads.make(name, reduced=True)
    ref = oracle.decode_workload(wl)
    check_decode(wl, run_decode(wl), ref, label=name)
    assert pa.pa_get_device_errors() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama_gqa_decode", "long_context_gqa", "fp8_kv", "mha_alibi_ragged"])
def test_full_size_workloads_sampled(name):
    wl = workloads.make(name)
    gpu = run_decode(wl)
    pairs = sample_pairs(wl, n=16 if name == "long_context_gqa" else 24)
    ref = oracle.decode_workload(wl, pairs=pairs)
    check_decode(wl, gpu, ref, pairs=pairs, label=name)
    # properties that hold at any size, on every row
    out, es, ml, tmp = gpu
    assert torch.isfinite(out.float()).all()
    lens = wl.seq_lens.to(torch.int64)
    P = es.shape[2]
    for s in range(wl.num_seqs):
        Ps = int(-(-int(lens[s]) // 512))
        assert torch.all(es[s, :, Ps:] == 0) and torch.all(ml[s, :, Ps:] == -float("inf"))
        if Ps:
            assert torch.all(es[s, :, :Ps] >= 1.0 - 1e-5)
    assert pa.pa_get_device_errors() == 0


EDGE_LENS = [0, 1, 2, 15, 16, 17, 511, 512, 513, 1024, 1025, 1536, 2047]


@pytest.mark.parametrize("d", [64, 80, 96, 112, 120, 128, 192, 256])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_head_and_block_sizes(d, bs):
    wl = workloads.build(num_seqs=len(EDGE_LENS), num_heads=8, num_kv_heads=2, head_size=d,
                         block_size=bs, seq_lens=EDGE_LENS, seed=100 + d + bs)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"d{d} bs{bs}")


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
def test_gqa_ratios(G):
    Hk = 2
    wl = workloads.build(num_seqs=3, num_heads=G * Hk, num_kv_heads=Hk, head_size=128,
                         block_size=16, seq_lens=[700, 33, 1500], seed=200 + G)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"G{G}")


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("kv", ["auto", "fp8_e4m3"])
@pytest.mark.parametrize("alibi", [False, True])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_dtypes_alibi(q_dtype, kv, alibi, bs):
    wl = workloads.build(num_seqs=5, num_heads=12, num_kv_heads=3, head_size=128, block_size=bs,
                         seq_lens=[1, 517, 1030, 64, 2500], q_dtype=q_dtype, kv_cache_dtype=kv,
                         alibi=alibi, k_scale=0.05 if kv != "auto" else 1.0,
                         v_scale=0.07 if kv != "auto" else 1.0, seed=300 + bs)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"{q_dtype} {kv} alibi={alibi}")


def test_non_unit_scales_on_half_cache():
    wl = workloads.build(num_seqs=3, num_heads=8, num_kv_heads=8, head_size=96, block_size=16,
                         seq_lens=[800, 1, 129], k_scale=0.5, v_scale=2.0, seed=11)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label="scales")


def test_alibi_long_positions_bf16():
    # absolute positions up to 32K with the steepest slopes: fp32 rounding of s_t would eat
    # the tolerance if the bias were applied at absolute positions inside the kernel
    wl = workloads.build(num_seqs=3, num_heads=16, num_kv_heads=16, head_size=96, block_size=32,
                         seq_lens=[32768, 20001, 513], q_dtype="bf16", alibi=True, seed=12)
    pairs = np.array([(s, h) for s in range(3) for h in (0, 1, 2, 7, 15)], dtype=np.int32)
    ref = oracle.decode_workload(wl, pairs=pairs)
    check_decode(wl, run_decode(wl), ref, pairs=pairs, label="alibi-long")


def test_extra_unused_partitions_and_wide_table():
    wl = workloads.build(num_seqs=4, num_heads=8, num_kv_heads=4, head_size=64, block_size=16,
                         seq_lens=[3, 700, 0, 1200], max_seq_len=4000, table_width=300, seed=13)
    ref = oracle.decode_workload(wl)
    gpu = run_decode(wl, max_num_partitions=9)
    # the oracle reports 8 partitions for max_seq_len 4000; the ninth must still be -inf / 0
    check_decode(wl, (gpu[0], gpu[1][:, :, :8], gpu[2][:, :, :8], gpu[3][:, :, :8]), ref, label="wide")
    assert torch.all(gpu[1][:, :, 8] == 0) and torch.all(gpu[2][:, :, 8] == -float("inf"))


def test_out_of_range_block_ids_are_masked_and_flagged():
    wl = workloads.build(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                         seq_lens=[100, 40], seed=14)
    bad = wl.block_tables.clone()
    bad[0, 2] = wl.num_blocks + 5  # tokens 32..47 of sequence 0 point outside the cache
    bad[1, 0] = -3                 # tokens 0..15 of sequence 1
    gpu = run_decode(workloads.Workload(**{**wl.__dict__, "block_tables": bad}))
    assert pa.pa_get_device_errors() & 1
    # Without ALiBi attention does not depend on token order, so masking a page must equal
    # attention over the sequence with that page removed.
    t = wl.block_tables
    ref_tables = torch.stack([torch.cat([t[0, :2], t[0, 3:7]]),
                              torch.cat([t[1, 1:3], t[1, 1:5]])]).to(torch.int32)
    wl_ref = workloads.Workload(**{**wl.__dict__, "block_tables": ref_tables,
                                   "seq_lens": torch.tensor([84, 24], dtype=torch.int32),
                                   "max_seq_len": 100})
    check_decode(wl_ref, gpu, oracle.decode_workload(wl_ref), label="masked pages")


def test_decode_is_deterministic():
    wl = workloads.make("llama_gqa_decode", reduced=True)
    dev = to_device(wl)
    a = run_decode(wl, dev)
    b = run_decode(wl, dev)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("name", ["llama_gqa_decode", "long_context_gqa", "fp8_kv", "mha_alibi_ragged"])
def test_tmp_output_in_query_dtype(name):
    # the pages' forward_decode keeps tmp_output in the output dtype
    wl = workloads.make(name, reduced=True)
    gpu = run_decode(wl, tmp_dtype=wl.query.dtype)
    assert gpu[3].dtype == wl.query.dtype
    check_decode(wl, gpu, oracle.decode_workload(wl), label=f"tmp16 {name}")


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
def test_output_only_four_byte_aligned(q_dtype):
    # the ABI asks 4-byte alignment of the output: an output that starts 4 bytes past an
    # 8-byte boundary takes the element-store path of the epilogue (one-partition sequences
    # write it directly)
    wl = workloads.build(num_seqs=3, num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                         seq_lens=[300, 1, 1500], q_dtype=q_dtype, seed=71)
    ref = oracle.decode_workload(wl)
    dev = {k: v for k, v in (("query", wl.query.cuda()), ("key_cache", wl.key_cache.cuda()),
                             ("value_cache", wl.value_cache.cuda()), ("block_tables", wl.block_tables.cuda()),
                             ("seq_lens", wl.seq_lens.cuda()))}
    S, H, d = wl.query.shape
    P = wl.max_num_partitions
    buf = torch.full((S * H * d + 2,), float("nan"), dtype=wl.query.dtype, device="cuda")
    out = buf[2:].view(S, H, d)  # 4 bytes past the allocation's start
    assert out.data_ptr() % 8 == 4
    es = torch.empty((S, H, P), dtype=torch.float32, device="cuda")
    ml = torch.empty_like(es)
    tmp = torch.empty((S, H, P, d), dtype=torch.float32, device="cuda")
    pa.pa_v2_decode(out, es, ml, tmp, dev["query"], dev["key_cache"], dev["value_cache"], wl.num_kv_heads, wl.scale,
                    dev["block_tables"], dev["seq_lens"], wl.block_size, wl.max_seq_len)
    torch.cuda.synchronize()
    check_decode(wl, (out.cpu(), es.cpu(), ml.cpu(), tmp.cpu()), ref, label=f"4-byte aligned output {q_dtype}")
