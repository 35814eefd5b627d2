"""GPU: pa_v2_decode_noalloc, the entry point for callers that cannot allocate device memory
(a plugin handed only a stream and a fixed budget), gives the same output as pa_v2_decode
with a caller-owned fp32 workspace (bit for bit: the same kernels run) and matches the fp64
oracle, on two calls in a row (the second call reuses scratch the first one left behind),
including the full long-context step that fills 19.4 MB of the scratch.

This file is named to be collected last, so a run that stops at its first failure has run
every other test before it; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import TOL_OUT, half_ulp, run_decode, sample_pairs, to_device

pytestmark = pytest.mark.gpu


def _noalloc_raw(wl, dev, out, max_seq_len=None):
    """Call the C entry point directly with raw device pointers; returns the status."""
    lib = pa.load()
    P = ctypes.c_void_p
    S, H, d = wl.query.shape
    msl = wl.max_seq_len if max_seq_len is None else max_seq_len
    return lib.pa_v2_decode_noalloc(
        P(out.data_ptr()), P(dev["query"].data_ptr()), P(dev["key_cache"].data_ptr()),
        P(dev["value_cache"].data_ptr()), S, H, wl.num_kv_heads, d, wl.scale,
        P(dev["block_tables"].data_ptr()), wl.block_tables.shape[1], wl.num_blocks,
        P(dev["seq_lens"].data_ptr()), wl.block_size, msl,
        None if dev["alibi"] is None else P(dev["alibi"].data_ptr()),
        pa.PA_DT_BF16 if wl.q_dtype == "bf16" else pa.PA_DT_F16,
        pa.PA_KV_FP8_E4M3 if wl.kv_cache_dtype == "fp8_e4m3" else pa.PA_KV_AUTO,
        wl.k_scale, wl.v_scale, P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["tiny", "llama_gqa_decode", "long_context_gqa", "fp8_kv", "mha_alibi_ragged"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    wl = workloads.make(name, reduced=True)
    dev = to_device(wl)
    # same kernels and launch as pa_v2_decode with an fp32 workspace: bit-identical output
    ref_gpu = run_decode(wl, dev, tmp_dtype=torch.float32)[0]
    ref = oracle.decode_workload(wl)["out"].reshape(wl.query.shape)
    allow = TOL_OUT[wl.kv_cache_dtype] + half_ulp(ref, wl.q_dtype)
    for call in range(2):
        out = torch.full(wl.query.shape, float("nan"), dtype=wl.query.dtype, device="cuda")
        st = _noalloc_raw(wl, dev, out)
        assert st == 0, f"call {call}: status {st} ({pa.STATUS.get(st)})"
        torch.cuda.synchronize()
        assert torch.equal(out.cpu().view(torch.int16), ref_gpu.view(torch.int16)), f"call {call}: differs"
        got = out.cpu().double().numpy()
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        err = np.abs(got - ref)
        assert (err <= allow).all(), f"call {call}: max error {err.max():.3g} against the oracle"


@pytest.mark.slow
def test_noalloc_full_long_context_against_the_oracle():
    # 4 sequences x 24 heads x head size 256 at 100K tokens: 19.4 MB of the fixed scratch
    wl = workloads.make("long_context_gqa")
    dev = to_device(wl)
    pairs = sample_pairs(wl, n=12)
    ref = oracle.decode_workload(wl, pairs=pairs)["out"]
    for call in range(2):
        out = torch.full(wl.query.shape, float("nan"), dtype=wl.query.dtype, device="cuda")
        assert _noalloc_raw(wl, dev, out) == 0
        torch.cuda.synchronize()
        got = out.cpu().double().numpy()[pairs[:, 0], pairs[:, 1]]
        err = np.abs(got - ref)
        assert (err <= TOL_OUT["auto"] + half_ulp(ref, wl.q_dtype)).all(), f"call {call}: {err.max():.3g}"


def test_noalloc_rejects_a_step_larger_than_its_scratch():
    # 64 sequences x 32 heads x 128 at 64K tokens needs ~256 MiB of workspace: refused
    # before anything is enqueued.
    wl = workloads.build(num_seqs=64, num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                         seq_lens=[17] * 64, max_seq_len=65536, table_width=4096, seed=3)
    dev = to_device(wl)
    out = torch.zeros(wl.query.shape, dtype=wl.query.dtype, device="cuda")
    assert _noalloc_raw(wl, dev, out) == 4  # PA_ERR_SCRATCH_TOO_SMALL
    assert torch.all(out == 0)
