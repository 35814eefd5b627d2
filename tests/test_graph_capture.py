"""GPU: the decode entry points captured in a CUDA graph and replayed.

A serving loop captures its decode step once per batch shape and replays it every step.
A graph freezes what the library chooses on the host (grid, partitions per CTA, kernel
form, cluster split), all of which follow from the call's sizes (num_seqs, heads, head
size, block size, max_seq_len, dtypes); the kernels read sequence lengths, block tables,
queries, new rows and caches from device memory at every replay.  Checked for each entry
point: after a second workload's inputs are copied into the captured buffers, a replay
gives bit for bit what an eager call on those inputs gives (output, partition statistics,
caches) and agrees with the fp64 oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import TOL_OUT, check_decode, half_ulp
from test_parity_append import oracle_append

pytestmark = pytest.mark.gpu

SHAPE = dict(num_seqs=6, num_heads=16, num_kv_heads=4, head_size=128, block_size=16, num_blocks=800,
             max_seq_len=4096, table_width=256)
LENS = ([4000, 1, 513, 2900, 0, 1700], [12, 3333, 4096, 512, 600, 1])
INPUTS = ("query", "key_cache", "value_cache", "block_tables", "seq_lens", "new_key", "new_value", "slot_mapping")


@pytest.fixture(autouse=True)
def _clear_device_errors():
    pa.pa_get_device_errors(reset=True)
    yield
    assert pa.pa_get_device_errors() == 0


def _pair(q_dtype, kv, alibi):
    scales = dict(k_scale=0.05, v_scale=0.07) if kv == "fp8_e4m3" else {}
    return [workloads.build(**SHAPE, seq_lens=lens, q_dtype=q_dtype, kv_cache_dtype=kv, alibi=alibi,
                            seed=700 + i, **scales) for i, lens in enumerate(LENS)]


class Step:
    """Device buffers of one decode step, the ones a captured graph reads and writes."""

    def __init__(self, wl, entry):
        self.wl, self.entry = wl, entry
        self.t = {k: getattr(wl, k).cuda().clone() for k in INPUTS}
        self.slopes = None if wl.alibi_slopes is None else wl.alibi_slopes.cuda()
        S, H, d = wl.query.shape
        self.es, self.ml, self.tmp = pa.workspace(S, H, d, wl.max_seq_len, "cuda")
        self.out = torch.empty_like(self.t["query"])
        self.order = torch.empty(S, dtype=torch.int32, device="cuda") if entry == "append_order" else None
        self.ctr = pa.decode_counters(S, H, wl.num_kv_heads, "cuda") if entry == "fused" else None

    def load(self, wl):
        for k in INPUTS:
            self.t[k].copy_(getattr(wl, k))
        for t in (self.out, self.es, self.ml):
            t.fill_(float("nan"))

    def __call__(self):
        t, wl = self.t, self.wl
        common = (wl.num_kv_heads, wl.scale)
        tail = (wl.block_size, wl.max_seq_len, self.slopes, wl.kv_cache_dtype, wl.k_scale, wl.v_scale)
        if self.entry.startswith("append"):
            pa.pa_v2_decode_append(self.out, self.es, self.ml, self.tmp, t["query"], t["new_key"], t["new_value"],
                                   t["key_cache"], t["value_cache"], *common, t["block_tables"], t["seq_lens"],
                                   *tail, order=self.order)
            return
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["key_cache"], t["value_cache"], t["slot_mapping"],
                                wl.kv_cache_dtype, wl.k_scale, wl.v_scale)
        if self.entry == "noalloc":
            pa.pa_v2_decode_noalloc(self.out, t["query"], t["key_cache"], t["value_cache"], *common,
                                    t["block_tables"], t["seq_lens"], *tail)
            return
        pa.pa_v2_decode(self.out, self.es, self.ml, self.tmp, t["query"], t["key_cache"], t["value_cache"], *common,
                        t["block_tables"], t["seq_lens"], *tail, counters=self.ctr)

    def results(self):
        r = [self.out, self.t["key_cache"], self.t["value_cache"]]
        if self.entry != "noalloc":
            r += [self.es, self.ml]
        return [x.cpu() for x in r]


def _bits(t):
    return t.view(torch.uint8) if t.dtype in (torch.uint8, torch.float8_e4m3fn) else \
        t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _same(a, b, label):
    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(_bits(x), _bits(y)), f"{label}: result {i} differs"


def _eager(step, wl):
    step.load(wl)
    step()
    torch.cuda.synchronize()
    return step.results()


def _check_oracle(wl, step, res, label):
    kr, vr, ref = oracle_append(wl)
    out = res[0]
    for name, got, want in (("key", res[1], kr), ("value", res[2], vr)):
        want = want.view(np.uint8) if want.dtype == np.uint8 else want.view(np.int16)
        assert np.array_equal(_bits(got).numpy(), want), f"{label}: {name} cache"
    if step.entry == "noalloc":
        r = ref["out"].reshape(out.shape)
        allow = TOL_OUT[wl.kv_cache_dtype] + half_ulp(r, wl.q_dtype)
        assert (np.abs(out.double().numpy() - r) <= allow).all(), f"{label}: output against the oracle"
        return
    es, ml = res[3], res[4]
    check_decode(wl, (out, es, ml, torch.zeros(0)), ref, label=label, check_tmp=False)


@pytest.mark.parametrize("entry", ["append", "append_order", "two_kernel", "fused", "noalloc"])
@pytest.mark.parametrize("q_dtype,kv,alibi", [("f16", "auto", False), ("bf16", "fp8_e4m3", True)])
def test_replay_matches_eager_and_oracle(entry, q_dtype, kv, alibi):
    if entry == "noalloc" and kv != "auto":
        kv, alibi = "auto", True  # the no-allocation entry takes per-tensor scales: keep it simple
    wl1, wl2 = _pair(q_dtype, kv, alibi)
    step = Step(wl1, entry)
    e1, e2 = _eager(step, wl1), _eager(step, wl2)  # eager first: per-kernel attributes are set
    step.load(wl1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for wl, ref, tag in ((wl1, e1, "first"), (wl2, e2, "second"), (wl1, e1, "first again")):
        step.load(wl)
        g.replay()
        torch.cuda.synchronize()
        res = step.results()
        _same(res, ref, f"{entry} {q_dtype} {kv}: {tag} inputs, replay against eager")
    _check_oracle(wl2, step, e2, f"{entry} {q_dtype} {kv} second inputs")


def test_two_replays_in_a_row_on_ping_pong_buffers():
    # two captured steps on two buffer sets, replayed alternately without a synchronisation
    # between them (the serving loop's pattern); the append entry leaves no state behind that
    # the next replay would read
    wl1, wl2 = _pair("bf16", "auto", True)
    steps = [Step(wl1, "append_order"), Step(wl2, "append_order")]
    refs = [_eager(steps[0], wl1), _eager(steps[1], wl2)]
    graphs = []
    for s, wl in zip(steps, (wl1, wl2)):
        s.load(wl)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            s()
        graphs.append(g)
    for rep in range(3):
        for s, wl in zip(steps, (wl1, wl2)):
            s.load(wl)
        graphs[0].replay()
        graphs[1].replay()
        torch.cuda.synchronize()
        for i, s in enumerate(steps):
            _same(s.results(), refs[i], f"replay round {rep} step {i}")


def _capture(fn):
    fn()  # uncaptured first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_copy_blocks_replay_reads_the_mapping_at_replay():
    # the mapping lives on the device: a replay copies the pairs the buffer holds then
    gen = torch.Generator().manual_seed(5)
    NB, layers = 40, 3
    kcs = [torch.randint(0, 255, (NB, 2, 8, 16, 16), generator=gen, dtype=torch.uint8).cuda() for _ in range(layers)]
    vcs = [torch.randint(0, 255, (NB, 2, 128, 16), generator=gen, dtype=torch.uint8).cuda() for _ in range(layers)]
    m = torch.tensor([[1, 2], [3, 4]], dtype=torch.int64, device="cuda")
    g = _capture(lambda: pa.pa_copy_blocks(kcs, vcs, m))
    for pairs in ([[5, 6], [7, 8]], [[30, 0], [12, 39]]):
        want = [t.cpu().numpy().copy() for t in kcs + vcs]
        mm = torch.tensor(pairs, dtype=torch.int64)
        for a in want:
            oracle.copy_blocks(a, a, mm)
        m.copy_(mm)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(kcs + vcs, want):
            assert np.array_equal(a.cpu().numpy(), b)


def test_swap_blocks_replay_moves_the_captured_pairs():
    # the mapping is read on the host when the call is made: a replay repeats the captured
    # pairs, with whatever the source blocks hold then
    gen = torch.Generator().manual_seed(6)
    src = torch.randint(0, 255, (16, 4, 64, 16), generator=gen, dtype=torch.uint8).cuda()
    dst = torch.zeros((12, 4, 64, 16), dtype=torch.uint8).pin_memory()
    m = torch.tensor([[3, 0], [15, 11], [7, 5]], dtype=torch.int64)
    g = _capture(lambda: pa.pa_swap_blocks(src, dst, m))
    src.copy_(torch.randint(0, 255, src.shape, generator=gen, dtype=torch.uint8))
    want = dst.numpy().copy()
    oracle.copy_blocks(want, src.cpu().numpy(), m)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(dst.numpy(), want)


def test_prefix_replay_with_split_contexts():
    # contexts above 16K tokens are cut into parts (caller-owned workspace); a replay on a
    # second workload's lengths, tables and rows matches an eager call bit for bit and the
    # oracle
    from gpu_harness import check_prefix, prefix_to_device
    kw = dict(num_seqs=3, num_heads=8, num_kv_heads=2, head_size=128, block_size=16, query_lens=[100, 37, 64],
              q_dtype="bf16", table_width=1280)
    wl1 = workloads.build_prefix(context_lens=[20000, 0, 700], seed=1, **kw)
    wl2 = workloads.build_prefix(context_lens=[300, 18000, 5], seed=2, **kw)
    assert wl2.key_cache.shape[0] <= wl1.key_cache.shape[0]
    dev = prefix_to_device(wl1)
    S, H, Hk, d = 3, 8, 2, 128
    mql = 100
    ws = torch.empty(pa.prefix_workspace_size(S, H, Hk, d, mql, 8), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev["query"])

    def call():
        pa.pa_prefix(out, dev["query"], dev["key"], dev["value"], dev["key_cache"], dev["value_cache"],
                     dev["block_tables"], dev["query_start_loc"], dev["context_lens"], mql, scale=wl1.scale,
                     workspace=ws, max_splits=8)

    def load(wl):
        for k in ("query", "key", "value", "block_tables", "query_start_loc", "context_lens"):
            dev[k].copy_(getattr(wl, k))
        for k in ("key_cache", "value_cache"):
            dev[k][:getattr(wl, k).shape[0]].copy_(getattr(wl, k))
        out.fill_(float("nan"))

    eager = []
    for wl in (wl1, wl2):
        load(wl)
        call()
        torch.cuda.synchronize()
        eager.append(out.cpu())
    load(wl1)
    g = _capture(call)
    for wl, ref in ((wl1, eager[0]), (wl2, eager[1])):
        load(wl)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.cpu().view(torch.int16), ref.view(torch.int16))
    check_prefix(wl2, eager[1], oracle.prefix_workload(wl2), label="prefix replay, second inputs")
