"""GPU parity: one k_scale / v_scale per kv head (pa_v2_decode_head_scales,
pa_v2_decode_append_head_scales, pa_reshape_and_cache_head_scales) against the fp64 oracle.

The dequantisation of "paged_attention_v2_pytorch.py" (cache values times k_scale / v_scale)
is taken per kv head.  Checked: decode outputs and partition statistics within the decode
tolerances, the writer's cache bytes bit for bit, the fused append (output and caches), and
that scales equal across heads give bit-identical results to the per-tensor entry points.
A scale that is not finite and positive is flagged (device error bit 8).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import check_decode, run_decode, sample_pairs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_errors():
    pa.pa_get_device_errors(reset=True)
    yield


def _scales(n, seed, lo=0.01, hi=0.4):
    rng = np.random.default_rng(seed)
    return [float(np.float32(x)) for x in np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))]


def _codes(t: torch.Tensor) -> np.ndarray:
    return (t.view(torch.uint8) if t.dtype in (torch.uint8, torch.float8_e4m3fn) else t.view(torch.int16)).cpu().numpy()


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("alibi", [False, True])
def test_decode_fp8_head_scales(q_dtype, bs, alibi):
    Hk = 4
    wl = workloads.build(num_seqs=6, num_heads=16, num_kv_heads=Hk, head_size=128, block_size=bs,
                         seq_lens=[1, 511, 513, 1600, 0, 2900], q_dtype=q_dtype, kv_cache_dtype="fp8_e4m3",
                         alibi=alibi, k_scales=_scales(Hk, 1), v_scales=_scales(Hk, 2), seed=600 + bs)
    ref = oracle.decode_workload(wl)
    check_decode(wl, run_decode(wl), ref, label=f"head scales {q_dtype} bs{bs} alibi={alibi}")
    assert pa.pa_get_device_errors() == 0


@pytest.mark.parametrize("G,d,kv", [(1, 96, "auto"), (6, 256, "fp8_e4m3"), (12, 128, "auto"), (16, 64, "fp8_e4m3")])
def test_decode_head_scales_gqa_and_head_sizes(G, d, kv):
    # the pages apply the scales to any cache dtype, 16-bit caches included
    Hk = 3
    wl = workloads.build(num_seqs=3, num_heads=G * Hk, num_kv_heads=Hk, head_size=d, block_size=16,
                         seq_lens=[700, 33, 1500], q_dtype="bf16", kv_cache_dtype=kv,
                         k_scales=_scales(Hk, 3, 0.25, 2.0), v_scales=_scales(Hk, 4, 0.25, 2.0), seed=610 + G)
    ref = oracle.decode_workload(wl)
    check_decode(wl, run_decode(wl), ref, label=f"head scales G{G} d{d} {kv}")


@pytest.mark.parametrize("kv", ["auto", "fp8_e4m3"])
def test_equal_head_scales_match_per_tensor_bitwise(kv):
    wl = workloads.build(num_seqs=4, num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                         seq_lens=[3000, 1, 700, 2600], kv_cache_dtype=kv, alibi=True,
                         k_scale=0.05, v_scale=0.07, seed=620)
    a = run_decode(wl)
    wlh = workloads.Workload(**{**wl.__dict__, "k_scales": torch.full((2,), wl.k_scale, dtype=torch.float32),
                                "v_scales": torch.full((2,), wl.v_scale, dtype=torch.float32)})
    b = run_decode(wlh)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype != torch.float32 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype != torch.float32 else y.view(torch.int32))


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
def test_writer_head_scales_bit_exact(q_dtype):
    Hk = 4
    wl = workloads.build(num_seqs=7, num_heads=8, num_kv_heads=Hk, head_size=128, block_size=16,
                         seq_lens=[3, 40, 0, 17, 512, 1, 99], q_dtype=q_dtype, kv_cache_dtype="fp8_e4m3",
                         k_scales=_scales(Hk, 5, 0.002, 1.0), v_scales=_scales(Hk, 6, 0.002, 1.0), seed=630)
    kr, vr = oracle._np(wl.key_cache).copy(), oracle._np(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key, wl.new_value, q_dtype, kr, vr, "fp8_e4m3", wl.slot_mapping,
                             block_size=16, k_scale=wl.k_scales, v_scale=wl.v_scales)
    kc, vc = wl.key_cache.cuda(), wl.value_cache.cuda()
    pa.pa_reshape_and_cache_head_scales(wl.new_key.cuda(), wl.new_value.cuda(), kc, vc, wl.slot_mapping.cuda(),
                                        "fp8_e4m3", k_scales=wl.k_scales.cuda(), v_scales=wl.v_scales.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_codes(kc), kr) and np.array_equal(_codes(vc), vr)
    assert pa.pa_get_device_errors() == 0


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
def test_append_head_scales(q_dtype):
    Hk = 3
    wl = workloads.build(num_seqs=5, num_heads=12, num_kv_heads=Hk, head_size=128, block_size=16,
                         seq_lens=[1, 517, 1030, 64, 2500], q_dtype=q_dtype, kv_cache_dtype="fp8_e4m3", alibi=True,
                         k_scales=_scales(Hk, 7), v_scales=_scales(Hk, 8), seed=640)
    from test_parity_append import _check_all
    _check_all(wl, f"append head scales {q_dtype}")
    assert pa.pa_get_device_errors() == 0


@pytest.mark.slow
def test_fp8_batch_full_size_head_scales_sampled():
    # the fp8 batch's shape (128 sequences, U[512..8192], 32/8 heads) with a scale per head
    wl = workloads.make("fp8_kv", k_scales=_scales(8, 9, 0.03, 0.08), v_scales=_scales(8, 10, 0.03, 0.08))
    pairs = sample_pairs(wl, n=16)
    ref = oracle.decode_workload(wl, pairs=pairs)
    check_decode(wl, run_decode(wl), ref, pairs=pairs, label="fp8 batch head scales")


def test_invalid_head_scale_is_flagged():
    # a zero v_scale for kv head 1: its rows come out as zeros, the flag is raised, the other
    # head is unaffected
    wl = workloads.build(num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                         seq_lens=[100, 700], kv_cache_dtype="fp8_e4m3", k_scales=[0.05, 0.05],
                         v_scales=[0.07, 0.07], seed=650)
    wl.v_scales = torch.tensor([0.07, 0.0], dtype=torch.float32)  # the caches were built at 0.07
    out = run_decode(wl)[0]
    assert pa.pa_get_device_errors() & 256
    assert torch.all(out[:, 2:] == 0)
    good = workloads.Workload(**{**wl.__dict__, "k_scales": None, "v_scales": None, "k_scale": 0.05,
                                 "v_scale": 0.07})
    ref = oracle.decode_workload(good)["out"].reshape(out.shape)
    assert np.abs(out[:, :2].double().numpy() - ref[:, :2]).max() <= 2e-2 + 1e-3


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


@pytest.mark.parametrize("env", [{"PA_DECODE_PX": "2"}, {"PA_DECODE_SPLIT": "2"}])
def test_head_scales_with_strides_and_cluster_split(env):
    # the per-head kernel form with CTAs striding over partitions, and with a 2-CTA cluster
    # sharing each partition (the partners hand their rows to the first CTA)
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    specs = [dict(num_seqs=4, num_heads=16, num_kv_heads=4, head_size=128, block_size=16,
                  seq_lens=[3000, 1, 700, 2600], kv_cache_dtype="fp8_e4m3", alibi=True,
                  k_scales=_scales(4, 11), v_scales=_scales(4, 12), seed=660)]
    code = _CHILD.format(here=here, root=os.path.dirname(here), specs=specs)
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
