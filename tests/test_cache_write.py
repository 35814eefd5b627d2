"""GPU: the slot-mapping cache writer is bit-exact against the oracle writer, and one full
decode step (write the new token, then attend over it) matches the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa
import workloads
from gpu_harness import check_decode, run_decode

pytestmark = pytest.mark.gpu


def _codes(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous().cpu()
    return t.view(torch.uint8).numpy() if t.element_size() == 1 else t.view(torch.int16).numpy()


@pytest.mark.parametrize("q_dtype,kv", [("f16", "auto"), ("bf16", "auto"), ("f16", "fp8_e4m3"),
                                        ("bf16", "fp8_e4m3")])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("d", [64, 96, 120, 128, 256])
def test_writer_bit_exact(q_dtype, kv, bs, d):
    if kv == "fp8_e4m3" and d % 16:
        pytest.skip("fp8 caches need head_size % 16 == 0")
    wl = workloads.build(num_seqs=9, num_heads=8, num_kv_heads=4, head_size=d, block_size=bs,
                         seq_lens=[1, 2, 0, 17, 512, 513, 33, 100, 7], q_dtype=q_dtype,
                         kv_cache_dtype=kv, k_scale=0.05 if kv != "auto" else 1.0,
                         v_scale=0.03 if kv != "auto" else 1.0, sigma=3.0, seed=d + bs)
    storage = wl.kv_storage
    kc_ref = _codes(wl.key_cache).copy()
    vc_ref = _codes(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key, wl.new_value, q_dtype, kc_ref, vc_ref, storage,
                             wl.slot_mapping, block_size=bs, k_scale=wl.k_scale, v_scale=wl.v_scale)
    kc = wl.key_cache.cuda()
    vc = wl.value_cache.cuda()
    pa.pa_reshape_and_cache(wl.new_key.cuda(), wl.new_value.cuda(), kc, vc, wl.slot_mapping.cuda(),
                            kv, wl.k_scale, wl.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(_codes(kc), kc_ref)
    assert np.array_equal(_codes(vc), vc_ref)
    assert pa.pa_get_device_errors() == 0


def test_writer_fp8_saturation_rounding_and_signed_zero():
    # hand-picked values around the e4m3 grid: ties, the saturation edge, infinities, signed zero
    vals = [448.0, 464.0, 500.0, -1e6, 2 ** -10, 3 * 2 ** -10, 15 * 2 ** -10, 1.0625, 1.1875,
            -0.0, 0.0, 431.99, 432.0, float("inf"), float("-inf"), 1e-30]
    d, Hk, bs = 64, 1, 16
    row = torch.zeros(d, dtype=torch.float32)
    row[:len(vals)] = torch.tensor(vals)
    key = row.to(torch.float16).view(1, Hk, d)
    value = (-row).to(torch.float16).view(1, Hk, d)
    kc = torch.zeros((2, Hk, d // 16, bs, 16), dtype=torch.uint8)
    vc = torch.zeros((2, Hk, d, bs), dtype=torch.uint8)
    slots = torch.tensor([bs + 3], dtype=torch.int64)
    kr, vr = kc.numpy().copy(), vc.numpy().copy()
    oracle.reshape_and_cache(key, value, "f16", kr, vr, "fp8_e4m3", slots, block_size=bs)
    kg, vg = kc.cuda(), vc.cuda()
    pa.pa_reshape_and_cache(key.cuda(), value.cuda(), kg, vg, slots.cuda(), "fp8_e4m3", 1.0, 1.0)
    torch.cuda.synchronize()
    assert np.array_equal(kg.cpu().numpy(), kr)
    assert np.array_equal(vg.cpu().numpy(), vr)


def test_writer_strided_rows_and_skipped_slots():
    # key/value as views into a fused qkv buffer (token stride > Hk * d), negative slots skipped
    T, H, Hk, d, bs = 6, 8, 2, 128, 16
    qkv = torch.randn(T, (H + 2 * Hk) * d, dtype=torch.float32).to(torch.float16)
    key = qkv[:, H * d:(H + Hk) * d].view(T, Hk, d)
    value = qkv[:, (H + Hk) * d:].view(T, Hk, d)
    kc = torch.randn(8, Hk, d // 8, bs, 8).to(torch.float16)
    vc = torch.randn(8, Hk, d, bs).to(torch.float16)
    slots = torch.tensor([5, -1, 17, 127, -7, 64], dtype=torch.int64)
    kr, vr = _codes(kc).copy(), _codes(vc).copy()
    oracle.reshape_and_cache(key.contiguous(), value.contiguous(), "f16", kr, vr, "f16", slots,
                             block_size=bs)
    kg, vg = kc.cuda(), vc.cuda()
    qkv_g = qkv.cuda()
    pa.pa_reshape_and_cache(qkv_g[:, H * d:(H + Hk) * d].view(T, Hk, d),
                            qkv_g[:, (H + Hk) * d:].view(T, Hk, d), kg, vg, slots.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_codes(kg), kr)
    assert np.array_equal(_codes(vg), vr)


def test_writer_flags_out_of_range_slot():
    kc = torch.zeros((2, 1, 8, 16, 8), dtype=torch.float16, device="cuda")
    vc = torch.zeros((2, 1, 64, 16), dtype=torch.float16, device="cuda")
    key = torch.ones((1, 1, 64), dtype=torch.float16, device="cuda")
    pa.pa_get_device_errors(reset=True)
    pa.pa_reshape_and_cache(key, key, kc, vc, torch.tensor([32], dtype=torch.int64, device="cuda"))
    assert pa.pa_get_device_errors() & 8
    assert torch.all(kc == 0) and torch.all(vc == 0)


@pytest.mark.parametrize("name", ["llama_gqa_decode", "fp8_kv", "mha_alibi_ragged"])
def test_full_decode_step_write_then_attend(name):
    wl = workloads.make(name, reduced=True)
    # oracle: write the step's new token into a copy of the cache, then decode
    kc_ref = oracle._np(wl.key_cache).copy()
    vc_ref = oracle._np(wl.value_cache).copy()
    oracle.reshape_and_cache(wl.new_key, wl.new_value, wl.q_dtype, kc_ref, vc_ref, wl.kv_storage,
                             wl.slot_mapping, block_size=wl.block_size, k_scale=wl.k_scale,
                             v_scale=wl.v_scale)
    ref = oracle.decode_workload(wl, key_cache=kc_ref, value_cache=vc_ref)
    # GPU: the same two calls on one stream
    from gpu_harness import to_device
    dev = to_device(wl)
    pa.pa_reshape_and_cache(wl.new_key.cuda(), wl.new_value.cuda(), dev["key_cache"], dev["value_cache"],
                            wl.slot_mapping.cuda(), wl.kv_cache_dtype, wl.k_scale, wl.v_scale)
    gpu = run_decode(wl, dev)
    check_decode(wl, gpu, ref, label=f"step {name}")
    assert np.array_equal(_codes(dev["key_cache"]), kc_ref)
