"""GPU: pa_v2_decode reads its inputs only after the kernel before it on the stream is done.

The decode kernels are launched with programmatic dependent launch, so their CTAs can start
while the previous kernel in the stream is still finishing.  A serving loop typically writes
the step's block tables and lengths with a kernel of its own just before the decode; the
decode must see those writes.  Here one elementwise kernel rewrites both (they share one
buffer) immediately before every decode call, alternating between two table sets that give
different results, and every call must match the oracle on the tables just written.
"""
from __future__ import annotations

import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import check_decode

pytestmark = pytest.mark.gpu


def _variant(wl, order):
    """The workload with its sequences' tables and lengths taken in `order` (the query rows
    stay put), so that each query row attends to another sequence's keys and values."""
    return workloads.Workload(**{**wl.__dict__, "block_tables": wl.block_tables[order].contiguous(),
                                 "seq_lens": wl.seq_lens[order].contiguous()})


@pytest.mark.parametrize("name", ["llama_gqa_decode", "mha_alibi_ragged"])
def test_tables_written_by_the_previous_kernel_are_seen(name):
    wl = workloads.make(name, reduced=True)
    S, H, d = wl.query.shape
    W = wl.block_tables.shape[1]
    order = torch.arange(S - 1, -1, -1)
    variants = [wl, _variant(wl, order)]
    refs = [oracle.decode_workload(v) for v in variants]

    # tables and lengths in one int32 buffer, so one kernel writes both
    def packed(v):
        return torch.cat([v.block_tables.reshape(-1), v.seq_lens]).to(torch.int32).cuda()

    sources = [packed(v) for v in variants]
    buf = torch.empty_like(sources[0])
    bt, sl = buf[: S * W].view(S, W), buf[S * W:]
    q, kc, vc = wl.query.cuda(), wl.key_cache.cuda(), wl.value_cache.cuda()
    slopes = None if wl.alibi_slopes is None else wl.alibi_slopes.cuda()
    es, ml, tmp = pa.workspace(S, H, d, wl.max_seq_len, "cuda")
    outs = []
    for i in range(6):
        out = torch.full_like(q, float("nan"))
        torch.mul(sources[i % 2], 1, out=buf)  # an elementwise kernel, right before the decode
        pa.pa_v2_decode(out, es, ml, tmp, q, kc, vc, wl.num_kv_heads, wl.scale, bt, sl, wl.block_size,
                        wl.max_seq_len, slopes, wl.kv_cache_dtype, wl.k_scale, wl.v_scale)
        outs.append((out, es.clone(), ml.clone(), tmp.clone()))
    torch.cuda.synchronize()
    for i, (out, e, m, t) in enumerate(outs):
        check_decode(variants[i % 2], (out.cpu(), e.cpu(), m.cpu(), t.cpu()), refs[i % 2],
                     label=f"{name} call {i}")
