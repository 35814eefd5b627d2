"""GPU parity: more than 8 query heads per kv head with 16-bit caches (the GQA view of
"paged_attention_v2_pytorch.py": query heads h * G .. h * G + G - 1 share kv head h).  The
grid then runs ceil(G / 8) CTAs per (partition, kv head), each serving up to 8 of the heads
over the same pages.

Checked against the fp64 oracle: G from 9 to 32 (partial last groups, two and four groups),
head sizes 64 to 128 including 120, block sizes 8/16/32, both query dtypes, ALiBi, edge
lengths, a 16-bit tmp_output, the fused append, the few-rows grid whose CTAs fold their
partitions into one row, and fp8 caches at G 8 to 16.  With 8 heads a CTA at head size 128
the library takes the kernel form whose warps pair up in the cross-warp reduction (three
CTAs an SM instead of two); the unpaired form is checked there too (PA_DECODE_PAIR=0), and
the paired one under 2- and 4-CTA clusters per partition and strided grids.
"""
from __future__ import annotations

import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import check_decode, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_errors():
    pa.pa_get_device_errors(reset=True)
    yield
    assert pa.pa_get_device_errors() == 0


@pytest.mark.parametrize("G", [9, 12, 16, 24, 32])
def test_gqa_ratios_above_eight(G):
    Hk = 2
    wl = workloads.build(num_seqs=3, num_heads=G * Hk, num_kv_heads=Hk, head_size=128, block_size=16,
                         seq_lens=[700, 33, 1500], seed=800 + G)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"G{G}")


@pytest.mark.parametrize("d", [64, 80, 96, 112, 120, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_head_sizes_and_block_sizes(d, bs):
    wl = workloads.build(num_seqs=4, num_heads=32, num_kv_heads=2, head_size=d, block_size=bs,
                         seq_lens=[1, 513, 1030, 2047], q_dtype="bf16", alibi=True, seed=820 + d + bs)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"G16 d{d} bs{bs}")


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("alibi", [False, True])
def test_dtypes_alibi_and_edge_lengths(q_dtype, alibi):
    wl = workloads.build(num_seqs=9, num_heads=28, num_kv_heads=2, head_size=128, block_size=16,
                         seq_lens=[0, 1, 15, 16, 17, 511, 512, 513, 3000], q_dtype=q_dtype, alibi=alibi,
                         seed=840)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"G14 {q_dtype} alibi={alibi}")


def test_sixteen_bit_tmp_output():
    wl = workloads.build(num_seqs=3, num_heads=32, num_kv_heads=2, head_size=96, block_size=32,
                         seq_lens=[2600, 700, 1], q_dtype="f16", alibi=True, seed=850)
    check_decode(wl, run_decode(wl, tmp_dtype=torch.float16), oracle.decode_workload(wl), label="G16 tmp16")


@pytest.mark.parametrize("G", [12, 16, 20])
def test_append(G):
    from test_parity_append import _check_all
    wl = workloads.build(num_seqs=4, num_heads=2 * G, num_kv_heads=2, head_size=128, block_size=16,
                         seq_lens=[1, 700, 2049, 4000], q_dtype="bf16", alibi=True, seed=860 + G)
    _check_all(wl, f"append G{G}")


def test_few_long_rows_fold_partitions():
    # 2 sequences x 2 kv heads of 40K tokens: fewer rows than CTA slots, so CTAs stream many
    # partitions and (append entry, tmp_output as scratch) fold them into one row each
    from test_parity_append import _check_all
    wl = workloads.build(num_seqs=2, num_heads=32, num_kv_heads=2, head_size=128, block_size=16,
                         seq_lens=[40000, 23456], q_dtype="f16", alibi=True, seed=870)
    _check_all(wl, "append G16 few rows")


@pytest.mark.parametrize("G,q_dtype,bs", [(8, "f16", 16), (8, "bf16", 32), (16, "bf16", 16), (12, "f16", 8)])
def test_fp8_cache(G, q_dtype, bs):
    wl = workloads.build(num_seqs=4, num_heads=2 * G, num_kv_heads=2, head_size=128, block_size=bs,
                         seq_lens=[1, 513, 1030, 3000], q_dtype=q_dtype, kv_cache_dtype="fp8_e4m3", k_scale=0.05,
                         v_scale=0.07, alibi=True, seed=890 + G)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"fp8 G{G} {q_dtype} bs{bs}")


_CHILD = r"""
import sys
sys.path.insert(0, {here!r}); sys.path.insert(0, {root!r})
import oracle, workloads
from gpu_harness import check_decode, run_decode
from test_parity_append import _check_all
for spec in {specs!r}:
    wl = workloads.build(**spec)
    check_decode(wl, run_decode(wl), oracle.decode_workload(wl), label=f"child decode {{spec}}")
    _check_all(wl, f"child append {{spec}}")
print("child ok")
"""


def test_unpaired_reduction_where_the_pairs_would_be_taken():
    # PA_DECODE_PAIR=0: 8-head CTAs at head size 128 keep one reduction row a warp (two CTAs
    # an SM); the paired form is what the library takes there by default
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    specs = [dict(num_seqs=4, num_heads=32, num_kv_heads=2, head_size=128, block_size=16,
                  seq_lens=[3000, 1, 700, 2600], q_dtype="bf16", alibi=True, seed=900),
             dict(num_seqs=3, num_heads=16, num_kv_heads=2, head_size=128, block_size=16,
                  seq_lens=[5000, 17, 1025], kv_cache_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.07, seed=901)]
    code = _CHILD.format(here=here, root=os.path.dirname(here), specs=specs)
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, PA_DECODE_PAIR="0"), capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


@pytest.mark.parametrize("env", [{"PA_DECODE_SPLIT": "2"}, {"PA_DECODE_SPLIT": "4"}, {"PA_DECODE_PX": "2"}])
def test_paired_reduction_with_cluster_split_and_strides(env):
    # the paired form under a 2- or 4-CTA cluster per partition (the partners hand their
    # summed rows to the first CTA) and with CTAs striding over partitions
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    specs = [dict(num_seqs=3, num_heads=32, num_kv_heads=2, head_size=128, block_size=16,
                  seq_lens=[3000, 1, 1400], q_dtype="f16", alibi=True, seed=910)]
    code = _CHILD.format(here=here, root=os.path.dirname(here), specs=specs)
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
