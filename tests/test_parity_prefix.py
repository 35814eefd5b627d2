"""GPU parity: pa_prefix (chunked-prefix attention, through the C ABI) against the fp64
oracle on the same seeded inputs.  Reduced chunked-prefill workloads are compared element
by element; the full-size ones (as the benchmark runs them) on sampled (token, head) rows
that include every chunk's first and last token and the 64-key tile edges.  Edge cases:
empty chunks and empty contexts, one-token chunks, contexts ending on and off tile and page
boundaries, every supported head size and block size, GQA ratios 1..16, strided q/k/v rows,
pages outside the cache (masked and flagged), contexts longer than the table (capped, as
the pages do) and NaN canaries in every cache slot the method must not read.  Contexts cut
into parts (the split path and its combine) are checked the same way, at part lengths down
to one 64-key tile and up to 32 parts."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import check_prefix, prefix_sample_rows, prefix_to_device, run_prefix

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_errors():
    pa.pa_get_device_errors(reset=True)
    yield


@pytest.mark.parametrize("name", list(workloads.PREFIX_CONFIGS))
def test_reduced_prefix_workloads_match_oracle(name):
    wl = workloads.make_prefix(name, reduced=True)
    check_prefix(wl, run_prefix(wl), oracle.prefix_workload(wl), label=name)
    assert pa.pa_get_device_errors() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefix_long_gqa", "prefix_llama_gqa"])
def test_full_size_prefix_sampled(name):
    # the binding's defaults, as the benchmark runs them (the library's plan: the long
    # workload's sequences each fill the GPU, so nothing is cut); the long workload also cut
    # into parts (an explicit split size)
    wl = workloads.make_prefix(name)
    rows = prefix_sample_rows(wl, n=40)
    ref = oracle.prefix_workload(wl, rows=rows)
    dev = prefix_to_device(wl)
    for max_splits, keys in (((None, 0), (8, 16384)) if name == "prefix_long_gqa" else ((None, 0),)):
        out = run_prefix(wl, dev, max_splits=max_splits, min_split_keys=keys)
        check_prefix(wl, out, ref, rows=rows, label=f"{name} max_splits={max_splits} min_split_keys={keys}")
        assert torch.isfinite(out.float()).all()
        assert pa.pa_get_device_errors() == 0


CTX = [0, 1, 63, 64, 65, 200, 511, 1000]
QL = [1, 0, 64, 65, 129, 3, 200, 17]


@pytest.mark.parametrize("d", [64, 80, 96, 112, 120, 128, 192, 256])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
def test_head_block_sizes_and_dtypes(d, bs, q_dtype):
    wl = workloads.build_prefix(num_seqs=len(CTX), num_heads=8, num_kv_heads=2, head_size=d,
                                block_size=bs, context_lens=CTX, query_lens=QL, q_dtype=q_dtype,
                                seed=500 + d + bs)
    check_prefix(wl, run_prefix(wl), oracle.prefix_workload(wl), label=f"d{d} bs{bs} {q_dtype}")


@pytest.mark.parametrize("G", [1, 2, 3, 5, 6, 7, 8, 16])
def test_gqa_ratios(G):
    wl = workloads.build_prefix(num_seqs=3, num_heads=2 * G, num_kv_heads=2, head_size=128, block_size=16,
                                context_lens=[300, 0, 77], query_lens=[90, 150, 1], seed=600 + G)
    check_prefix(wl, run_prefix(wl), oracle.prefix_workload(wl), label=f"G{G}")


def test_strided_rows():
    # q/k/v as views of wider rows (a fused qkv projection's output)
    wl = workloads.build_prefix(num_seqs=2, num_heads=8, num_kv_heads=2, head_size=64, block_size=16,
                                context_lens=[100, 33], query_lens=[70, 40], seed=700)
    out = run_prefix(wl, q_rows=8 * 64 + 64, kv_rows=2 * (2 * 64 + 16))
    check_prefix(wl, out, oracle.prefix_workload(wl), label="strided")


def test_max_query_len_larger_than_needed():
    wl = workloads.make_prefix("prefix_tiny")
    check_prefix(wl, run_prefix(wl, max_query_len=wl.max_query_len + 300), oracle.prefix_workload(wl),
                 label="wide grid")
    assert pa.pa_get_device_errors() == 0


def test_chunk_longer_than_max_query_len_is_skipped_and_flagged():
    wl = workloads.make_prefix("prefix_tiny")  # chunks of 5, 70, 129 tokens
    out = run_prefix(wl, max_query_len=100)
    assert pa.pa_get_device_errors() & 128
    qsl = wl.query_start_loc.tolist()
    assert torch.isnan(out[qsl[2]:qsl[3]].float()).all()  # the 129-token chunk is untouched
    ref = oracle.prefix_workload(wl)
    check_prefix(wl, out[:qsl[2]], ref[:qsl[2]], label="other chunks")


def test_out_of_range_page_is_masked_and_flagged():
    wl = workloads.build_prefix(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                                context_lens=[100, 40], query_lens=[20, 9], seed=800)
    bad = wl.block_tables.clone()
    bad[0, 2] = wl.num_blocks + 5  # context tokens 32..47 of sequence 0
    out = run_prefix(workloads.PrefixWorkload(**{**wl.__dict__, "block_tables": bad}))
    assert pa.pa_get_device_errors() & 32
    # attention has no positional term, so masking a page equals dropping its tokens
    t = wl.block_tables
    ref_tables = torch.stack([torch.cat([t[0, :2], t[0, 3:]]), t[1, :-1]]).to(torch.int32)
    ref_wl = workloads.PrefixWorkload(**{**wl.__dict__, "block_tables": ref_tables,
                                         "context_lens": torch.tensor([84, 40], dtype=torch.int32)})
    check_prefix(wl, out, oracle.prefix_workload(ref_wl), label="masked page")


def test_context_longer_than_table_is_capped_and_flagged():
    wl = workloads.build_prefix(num_seqs=1, num_heads=4, num_kv_heads=1, head_size=64, block_size=16,
                                context_lens=[64], query_lens=[10], table_width=5, seed=900)
    # a context of 200 tokens is capped to the table's 5 blocks = 80 tokens; slots 64..79
    # hold chunk canaries in this workload, so give that block real values first
    kc = wl.key_cache.clone()
    vc = wl.value_cache.clone()
    b = int(wl.block_tables[0, 4])
    g = torch.Generator().manual_seed(1)
    kc[b] = torch.randn(kc[b].shape, generator=g).to(kc.dtype)
    vc[b] = torch.randn(vc[b].shape, generator=g).to(vc.dtype)
    capped = workloads.PrefixWorkload(**{**wl.__dict__, "key_cache": kc, "value_cache": vc,
                                         "context_lens": torch.tensor([80], dtype=torch.int32)})
    over = workloads.PrefixWorkload(**{**capped.__dict__, "context_lens": torch.tensor([200], dtype=torch.int32)})
    out = run_prefix(over)
    assert pa.pa_get_device_errors() & 64
    check_prefix(wl, out, oracle.prefix_workload(capped), label="capped")


def test_prefix_is_deterministic():
    wl = workloads.make_prefix("prefix_llama_gqa", reduced=True)
    dev = prefix_to_device(wl)
    a = run_prefix(wl, dev)
    b = run_prefix(wl, dev)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_many_sequences_short_chunks():
    # 300 sequences (grid z), chunks of 0-40 new tokens over contexts of 0-700 tokens, bf16,
    # block size 32: most CTAs see one partial context tile and one causal chunk tile
    rng = np.random.default_rng(1100)
    S = 300
    ctx = rng.integers(0, 700, S).tolist()
    ql = rng.integers(0, 41, S).tolist()
    wl = workloads.build_prefix(num_seqs=S, num_heads=8, num_kv_heads=2, head_size=128, block_size=32,
                                context_lens=ctx, query_lens=ql, q_dtype="bf16", seed=1100)
    out = run_prefix(wl)
    rows = prefix_sample_rows(wl, n=80)
    check_prefix(wl, out, oracle.prefix_workload(wl, rows=rows), rows=rows, label="many seqs")
    assert pa.pa_get_device_errors() == 0


# ---- contexts cut into parts ----------------------------------------------------------------

def test_library_split_plan():
    # the library's plan cuts contexts only where one sequence's CTAs would fill less than half
    # the GPU: a few new tokens over a long context are cut, the long-context prefill is not
    assert pa.prefix_num_parts(24, 4, 256, torch.float16, 1024, 99328 // 16, 16) == 1
    n = pa.prefix_num_parts(32, 8, 128, torch.bfloat16, 64, 40960 // 16, 16)
    assert n == 3  # 40960 tokens in parts of at least 16384: up to 3
    assert pa.prefix_num_parts(32, 8, 128, torch.bfloat16, 64, 40960 // 16, 16, has_workspace=False) == 1
    wl = workloads.build_prefix(num_seqs=2, num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                                context_lens=[40000, 700], query_lens=[64, 9], q_dtype="bf16", seed=1190)
    out = run_prefix(wl)  # the binding takes a workspace and the library cuts the long context
    check_prefix(wl, out, oracle.prefix_workload(wl), label="library plan, cut")
    assert pa.pa_get_device_errors() == 0


@pytest.mark.parametrize("max_splits", [2, 3, 8, 32])
def test_split_contexts_match_oracle(max_splits):
    # parts as short as one 64-key tile: every context above 64 tokens is cut (up to 16 tiles
    # here, so 32 parts leaves one tile per part)
    wl = workloads.build_prefix(num_seqs=len(CTX), num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                context_lens=CTX, query_lens=QL, q_dtype="bf16", seed=1200 + max_splits)
    out = run_prefix(wl, max_splits=max_splits, min_split_keys=64)
    check_prefix(wl, out, oracle.prefix_workload(wl), label=f"max_splits={max_splits}")
    assert pa.pa_get_device_errors() == 0


@pytest.mark.parametrize("d,bs,q_dtype", [(64, 8, "f16"), (80, 16, "bf16"), (192, 32, "bf16"),
                                          (256, 16, "f16"), (256, 32, "bf16")])
def test_split_head_sizes(d, bs, q_dtype):
    # every tensor-memory plan (two S buffers, Q half in shared memory, one S buffer, P in
    # shared memory) through the partial-result epilogue
    ctx = [130, 640, 0, 64 * 9, 64 * 9 + 1, 1500]
    ql = [33, 70, 20, 1, 128, 9]
    wl = workloads.build_prefix(num_seqs=len(ctx), num_heads=8, num_kv_heads=2, head_size=d, block_size=bs,
                                context_lens=ctx, query_lens=ql, q_dtype=q_dtype, seed=1300 + d + bs)
    out = run_prefix(wl, max_splits=4, min_split_keys=128)
    check_prefix(wl, out, oracle.prefix_workload(wl), label=f"split d{d} bs{bs} {q_dtype}")
    assert pa.pa_get_device_errors() == 0


def test_split_and_unsplit_agree_closely():
    # the same inputs in one part and in parts: both within the oracle bar, and close to each
    # other (they differ only by fp32 summation order and the final rounding)
    wl = workloads.make_prefix("prefix_long_gqa", reduced=True)
    dev = prefix_to_device(wl)
    one = run_prefix(wl, dev, max_splits=1)
    parts = run_prefix(wl, dev, max_splits=5, min_split_keys=64)
    ref = oracle.prefix_workload(wl)
    check_prefix(wl, one, ref, label="one part")
    check_prefix(wl, parts, ref, label="parts")
    assert (one.float() - parts.float()).abs().max().item() <= 4e-3


def test_split_with_masked_page_and_capped_context():
    # a page outside the cache in the middle part, and a context longer than its table row
    wl = workloads.build_prefix(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                                context_lens=[400, 40], query_lens=[20, 9], seed=1400)
    bad = wl.block_tables.clone()
    bad[0, 10] = wl.num_blocks + 5  # context tokens 160..175 of sequence 0
    out = run_prefix(workloads.PrefixWorkload(**{**wl.__dict__, "block_tables": bad}), max_splits=4,
                     min_split_keys=64)
    assert pa.pa_get_device_errors() & 32
    t = wl.block_tables
    ref_tables = torch.stack([torch.cat([t[0, :10], t[0, 11:]]), t[1, :-1]]).to(torch.int32)
    ref_wl = workloads.PrefixWorkload(**{**wl.__dict__, "block_tables": ref_tables,
                                         "context_lens": torch.tensor([384, 40], dtype=torch.int32)})
    check_prefix(wl, out, oracle.prefix_workload(ref_wl), label="split masked page")

    wl = workloads.build_prefix(num_seqs=1, num_heads=4, num_kv_heads=1, head_size=64, block_size=16,
                                context_lens=[320], query_lens=[10], table_width=21, seed=1401)
    kc, vc = wl.key_cache.clone(), wl.value_cache.clone()
    b = int(wl.block_tables[0, 20])
    g = torch.Generator().manual_seed(2)
    kc[b] = torch.randn(kc[b].shape, generator=g).to(kc.dtype)
    vc[b] = torch.randn(vc[b].shape, generator=g).to(vc.dtype)
    capped = workloads.PrefixWorkload(**{**wl.__dict__, "key_cache": kc, "value_cache": vc,
                                         "context_lens": torch.tensor([336], dtype=torch.int32)})
    over = workloads.PrefixWorkload(**{**capped.__dict__, "context_lens": torch.tensor([1000], dtype=torch.int32)})
    out = run_prefix(over, max_splits=3, min_split_keys=64)
    assert pa.pa_get_device_errors() & 64
    check_prefix(wl, out, oracle.prefix_workload(capped), label="split capped")


def test_split_is_deterministic():
    wl = workloads.make_prefix("prefix_llama_gqa", reduced=True)
    dev = prefix_to_device(wl)
    a = run_prefix(wl, dev, max_splits=6, min_split_keys=64)
    b = run_prefix(wl, dev, max_splits=6, min_split_keys=64)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_auto_workspace_matches_explicit_workspace():
    # the binding's own workspace (torch allocator) and a caller-owned one give identical bits
    wl = workloads.make_prefix("prefix_long_gqa", reduced=True)
    dev = prefix_to_device(wl)
    auto = run_prefix(wl, dev, max_splits=4, min_split_keys=64)
    nbytes = pa.prefix_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size,
                                      wl.max_query_len, 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full(wl.query.shape, float("nan"), dtype=wl.query.dtype, device="cuda")
    pa.pa_prefix(out, dev["query"], dev["key"], dev["value"], dev["key_cache"], dev["value_cache"],
                 dev["block_tables"], dev["query_start_loc"], dev["context_lens"], wl.max_query_len,
                 scale=wl.scale, workspace=ws, max_splits=4, min_split_keys=64)
    torch.cuda.synchronize()
    assert torch.equal(auto.view(torch.int16), out.cpu().view(torch.int16))


def test_concurrent_calls_on_two_streams():
    # two split calls in flight at once on separate streams, each with its own workspace
    a = workloads.make_prefix("prefix_long_gqa", reduced=True)
    b = workloads.make_prefix("prefix_llama_gqa", reduced=True)
    da, db = prefix_to_device(a), prefix_to_device(b)
    oa = torch.full(a.query.shape, float("nan"), dtype=a.query.dtype, device="cuda")
    ob = torch.full(b.query.shape, float("nan"), dtype=b.query.dtype, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for wl, d, o, st in ((a, da, oa, sa), (b, db, ob, sb)):
        with torch.cuda.stream(st):
            pa.pa_prefix(o, d["query"], d["key"], d["value"], d["key_cache"], d["value_cache"], d["block_tables"],
                         d["query_start_loc"], d["context_lens"], wl.max_query_len, scale=wl.scale, stream=st,
                         max_splits=3, min_split_keys=64)
    torch.cuda.synchronize()
    check_prefix(a, oa.cpu(), oracle.prefix_workload(a), label="stream a")
    check_prefix(b, ob.cpu(), oracle.prefix_workload(b), label="stream b")
    assert pa.pa_get_device_errors() == 0


def test_timing_hook_brackets_the_attention_kernel():
    # events installed with pa_v2_set_timing_events are recorded around the prefix attention
    # kernel: positive, and no longer than the whole call (which adds the combine)
    wl = workloads.make_prefix("prefix_long_gqa", reduced=True)
    dev = prefix_to_device(wl)
    out = torch.empty_like(dev["query"])
    kb, ke = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cb, ce = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kb.record(); ke.record()  # create the events
    torch.cuda.synchronize()
    pa.pa_v2_set_timing_events(kb, ke)
    try:
        cb.record()
        pa.pa_prefix(out, dev["query"], dev["key"], dev["value"], dev["key_cache"], dev["value_cache"],
                     dev["block_tables"], dev["query_start_loc"], dev["context_lens"], wl.max_query_len,
                     scale=wl.scale, max_splits=4, min_split_keys=64)
        ce.record()
    finally:
        pa.pa_v2_set_timing_events(None, None)
    torch.cuda.synchronize()
    k_ms, c_ms = kb.elapsed_time(ke), cb.elapsed_time(ce)
    assert 0.0 < k_ms <= c_ms
