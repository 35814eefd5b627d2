"""GPU: block moves ("paged_attn.py" copy_blocks / swap_blocks) are bit-exact against the
oracle's block copy, across layers, dtypes and directions (GPU <-> pinned host)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_v2_gb300 as pa

pytestmark = pytest.mark.gpu


def _codes(t):
    t = t.contiguous().cpu()
    return t.view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.uint8])
@pytest.mark.parametrize("layers", [1, 3, 70])
def test_copy_blocks_bit_exact(dtype, layers):
    g = torch.Generator().manual_seed(layers)
    NB, Hk, d, bs = 48, 2, 64, 16
    x = 16 if dtype == torch.uint8 else 8
    def rand(shape):
        return torch.randint(0, 255, shape, generator=g, dtype=torch.uint8).view(dtype) if dtype != torch.uint8 \
            else torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
    kshape = (NB, Hk, d // x, bs, x * (2 if dtype != torch.uint8 else 1))
    vshape = (NB, Hk, d, bs * (2 if dtype != torch.uint8 else 1))
    kcs = [rand(kshape) for _ in range(layers)]
    vcs = [rand(vshape) for _ in range(layers)]
    perm = torch.randperm(NB, generator=g)
    m = torch.stack([perm[:10], perm[10:20]], dim=1).to(torch.int64)  # no dst is a src
    ref_k = [_codes(t).copy() for t in kcs]
    ref_v = [_codes(t).copy() for t in vcs]
    for a in ref_k + ref_v:
        oracle.copy_blocks(a, a, m)
    gk = [t.cuda() for t in kcs]
    gv = [t.cuda() for t in vcs]
    pa.pa_get_device_errors(reset=True)
    pa.pa_copy_blocks(gk, gv, m.cuda())
    torch.cuda.synchronize()
    for a, b in zip(gk + gv, ref_k + ref_v):
        assert np.array_equal(_codes(a), b)
    assert pa.pa_get_device_errors() == 0


def test_copy_blocks_flags_out_of_range_pairs():
    kc = torch.zeros((4, 1, 8, 16, 8), dtype=torch.float16, device="cuda")
    vc = torch.zeros((4, 1, 64, 16), dtype=torch.float16, device="cuda")
    kc[1] = 1.0
    pa.pa_get_device_errors(reset=True)
    pa.pa_copy_blocks([kc], [vc], torch.tensor([[1, 2], [0, 7]], dtype=torch.int64, device="cuda"))
    assert pa.pa_get_device_errors() & 16
    assert torch.all(kc[2] == 1.0) and torch.all(kc[0] == 0)


@pytest.mark.parametrize("direction", ["d2h", "h2d", "d2d"])
def test_swap_blocks_bit_exact(direction):
    g = torch.Generator().manual_seed(3)
    shape = (32, 4, 128, 16)
    src = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
    dst = torch.randint(0, 255, (20,) + shape[1:], generator=g, dtype=torch.uint8)
    m = torch.tensor([[3, 0], [31, 19], [7, 5], [0, 11]], dtype=torch.int64)
    want = dst.numpy().copy()
    oracle.copy_blocks(want, src.numpy(), m)
    s_dev = src.cuda() if direction in ("d2h", "d2d") else src.pin_memory()
    d_dev = dst.cuda() if direction in ("h2d", "d2d") else dst.pin_memory()
    pa.pa_swap_blocks(s_dev, d_dev, m)
    torch.cuda.synchronize()
    assert np.array_equal(d_dev.cpu().numpy(), want)


def test_swap_blocks_rejects_out_of_range_on_host():
    src = torch.zeros((4, 256), dtype=torch.uint8, device="cuda")
    dst = torch.zeros((4, 256), dtype=torch.uint8).pin_memory()
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_swap_blocks(src, dst, torch.tensor([[0, 4]], dtype=torch.int64))


@pytest.mark.parametrize("direction", ["h2d", "d2h"])
def test_swap_blocks_with_pageable_host_memory(direction):
    # host memory the device cannot address (not pinned): one copy per pair, same result
    g = torch.Generator().manual_seed(4)
    shape = (24, 2, 64, 16)
    src = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
    dst = torch.randint(0, 255, (16,) + shape[1:], generator=g, dtype=torch.uint8)
    m = torch.tensor([[5, 1], [23, 15], [0, 0]], dtype=torch.int64)
    want = dst.numpy().copy()
    oracle.copy_blocks(want, src.numpy(), m)
    s_dev = src if direction == "h2d" else src.cuda()
    d_dev = dst.cuda() if direction == "h2d" else dst
    pa.pa_swap_blocks(s_dev, d_dev, m)
    torch.cuda.synchronize()
    assert np.array_equal(d_dev.cpu().numpy(), want)


def test_swap_blocks_many_pairs_over_several_launches():
    # more pairs than one launch carries (480): every block moved, in both directions
    g = torch.Generator().manual_seed(5)
    NB = 1200
    src = torch.randint(0, 255, (NB, 2, 16, 16), generator=g, dtype=torch.uint8).cuda()
    host = torch.zeros((NB, 2, 16, 16), dtype=torch.uint8).pin_memory()
    perm = torch.randperm(NB, generator=g)
    m = torch.stack([perm[:1000], perm[200:1200]], 1).contiguous()
    want = host.numpy().copy()
    oracle.copy_blocks(want, src.cpu().numpy(), m)
    pa.pa_swap_blocks(src, host, m)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), want)
    back = torch.zeros_like(src)
    pa.pa_swap_blocks(host, back, m[:, [1, 0]].contiguous())
    torch.cuda.synchronize()
    want2 = np.zeros_like(want)
    oracle.copy_blocks(want2, host.numpy(), m[:, [1, 0]].contiguous())
    assert np.array_equal(back.cpu().numpy(), want2)
