"""CPU-only checks of the C-ABI library: it builds, loads, exports every function the
header declares, and rejects invalid arguments on the host before touching a device."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_v2_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa_v2.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for must in ("pa_v2_decode", "pa_reshape_and_cache", "pa_v2_partition_size", "pa_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib_path = pa._build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s(pa_\w+)$", out, flags=re.M))
    assert set(_declared()) <= exported, set(_declared()) - exported
    lib = ctypes.CDLL(lib_path)
    for name in _declared():
        assert hasattr(lib, name)


def test_partition_size_and_status_strings():
    assert pa.pa_v2_partition_size() == 512
    assert pa.pa_status_string(0) == "ok"
    assert pa.pa_status_string(1) == "invalid argument"
    assert pa.pa_status_string(2) == "unsupported combination"


def _decode_raw(**over):
    """Call pa_v2_decode with fake (never dereferenced) pointers; returns the status."""
    lib = pa.load()
    P = 0x10000  # 16-byte aligned fake address: validation must fail before any use
    a = dict(output=P, exp_sums=P, max_logits=P, tmp_output=P, query=P, key_cache=P, value_cache=P,
             num_seqs=2, num_heads=8, num_kv_heads=2, head_size=128, scale=0.088,
             block_tables=P, max_blocks_per_seq=64, num_blocks=100, seq_lens=P, block_size=16,
             max_seq_len=1024, max_num_partitions=2, alibi_slopes=None, q_dtype=0, kv=0, tmp=2,
             k_scale=1.0, v_scale=1.0)
    a.update(over)
    return lib.pa_v2_decode(a["output"], a["exp_sums"], a["max_logits"], a["tmp_output"], a["query"],
                            a["key_cache"], a["value_cache"], a["num_seqs"], a["num_heads"],
                            a["num_kv_heads"], a["head_size"], a["scale"], a["block_tables"],
                            a["max_blocks_per_seq"], a["num_blocks"], a["seq_lens"], a["block_size"],
                            a["max_seq_len"], a["max_num_partitions"], a["alibi_slopes"],
                            a["q_dtype"], a["kv"], a["tmp"], a["k_scale"], a["v_scale"], None)


@pytest.mark.parametrize("over,status", [
    (dict(num_heads=6, num_kv_heads=4), 1),          # H % Hk != 0
    (dict(block_size=24), 1),                        # 512 % bs != 0
    (dict(block_size=64), 2),                        # valid but not built
    (dict(head_size=100), 2),                        # not a supported head size
    (dict(head_size=120, kv=1), 1),                  # fp8 needs head_size % 16 == 0
    (dict(max_num_partitions=1), 1),                 # fewer partitions than max_seq_len needs
    (dict(max_blocks_per_seq=10), 1),                # table narrower than max_seq_len needs
    (dict(k_scale=0.0), 1),
    (dict(v_scale=-1.0), 1),
    (dict(k_scale=float("inf")), 1),
    (dict(scale=float("nan")), 1),
    (dict(output=None), 1),
    (dict(query=None), 1),
    (dict(tmp_output=None), 1),
    (dict(key_cache=0x10008), 1),                    # bulk copies need 16-byte alignment
    (dict(q_dtype=2), 2),                            # fp32 query not built
    (dict(tmp=1), 2),                                # tmp_output dtype other than fp32 / q
    (dict(kv=7), 1),
    (dict(num_blocks=0), 1),
    (dict(num_seqs=-1), 1),
    (dict(num_seqs=70000), 2),
    (dict(num_heads=8 * 70000, num_kv_heads=70000), 2),   # grid rows past 65535
])
def test_decode_rejects_invalid_arguments_on_host(over, status):
    assert _decode_raw(**over) == status


def test_decode_with_zero_sequences_is_a_noop():
    assert _decode_raw(num_seqs=0, output=None, query=None) == 0


def test_fused_decode_host_checks():
    lib = pa.load()
    P = 0x10000
    # one counter per (sequence, kv head, group of <= 8 query heads)
    assert pa.decode_num_counters(2, 8, 2) == 4
    assert pa.decode_num_counters(3, 32, 2) == 12        # 16 query heads per kv head: 2 groups
    assert pa.decode_num_counters(2, 6, 4) == 0          # H % Hk != 0
    args = [P, P, P, P, P, P, P, 2, 8, 2, 128, 0.088, P, 64, 100, P, 16, 1024, 2, None, 0, 0, 2, 1.0, 1.0]
    assert lib.pa_v2_decode_fused(*args, 0x10002, 4, None) == 1    # counters not 4-byte aligned
    assert lib.pa_v2_decode_fused(*args, P, 3, None) == 1          # fewer counters than the step needs
    bad = list(args)
    bad[9] = 3                                                     # H % Hk != 0, as pa_v2_decode
    assert lib.pa_v2_decode_fused(*bad, P, 4, None) == 1
    zero = list(args)
    zero[7] = 0                                                    # no sequences: nothing to do
    assert lib.pa_v2_decode_fused(*zero, None, 0, None) == 0


def test_head_scale_entry_points_host_checks():
    # arguments as the per-tensor entry points, with two device arrays in place of the floats;
    # every case below is rejected (or is a no-op) before anything touches the device
    lib = pa.load()
    P = 0x10000
    for name in ("pa_v2_decode_head_scales", "pa_v2_decode_append_head_scales", "pa_reshape_and_cache_head_scales"):
        assert name in _declared()
    dec = [P, P, P, P, P, P, P, 2, 8, 2, 128, 0.088, P, 64, 100, P, 16, 1024, 2, None, 0, 0, 2]
    assert lib.pa_v2_decode_head_scales(*dec, None, P, None) == 1          # no k_scales
    assert lib.pa_v2_decode_head_scales(*dec, P, None, None) == 1          # no v_scales
    assert lib.pa_v2_decode_head_scales(*dec, P + 2, P, None) == 1         # misaligned
    bad = list(dec)
    bad[9] = 3                                                             # H % Hk != 0
    assert lib.pa_v2_decode_head_scales(*bad, P, P, None) == 1
    zero = list(dec)
    zero[7] = 0
    assert lib.pa_v2_decode_head_scales(*zero, P, P, None) == 0            # no sequences
    app = [P, P, P, P, P, P, P, 256, 256, P, P, 2, 8, 2, 128, 0.088, P, 64, 100, P, 16, 1024, 2, None, 0, 0, 2]
    assert lib.pa_v2_decode_append_head_scales(*app, None, P, None, None) == 1
    assert lib.pa_v2_decode_append_head_scales(*app, P, P + 1, None, None) == 1
    assert lib.pa_v2_decode_append_head_scales(*app, P, P, P + 2, None) == 1   # misaligned order buffer
    short = list(app)
    short[7] = 100                                                         # key rows shorter than Hk * d
    assert lib.pa_v2_decode_append_head_scales(*short, P, P, None, None) == 1
    wr = [P, P, 256, 256, P, P, P, 4, 2, 128, 16, 10, 0, 1]
    assert lib.pa_reshape_and_cache_head_scales(*wr, None, P, None) == 1
    assert lib.pa_reshape_and_cache_head_scales(*wr, P, P + 2, None) == 1
    wr0 = list(wr)
    wr0[7] = 0
    assert lib.pa_reshape_and_cache_head_scales(*wr0, P, P, None) == 0     # no tokens


def test_order_entry_point_host_checks():
    lib = pa.load()
    P = 0x10000
    assert "pa_v2_decode_order" in _declared()
    assert lib.pa_v2_decode_order(P, -1, P, None) == 1          # negative count
    assert lib.pa_v2_decode_order(P, 65536, P, None) == 1       # beyond the grid's z extent
    assert lib.pa_v2_decode_order(None, 4, P, None) == 1
    assert lib.pa_v2_decode_order(P, 4, P + 2, None) == 1       # misaligned
    assert lib.pa_v2_decode_order(None, 0, None, None) == 0     # nothing to order


def _cache_raw(**over):
    lib = pa.load()
    P = 0x10000
    a = dict(key=P, value=P, ks=256, vs=256, key_cache=P, value_cache=P, slots=P, T=4, Hk=2, d=128,
             bs=16, nb=10, src=0, kv=0, k_scale=1.0, v_scale=1.0)
    a.update(over)
    return lib.pa_reshape_and_cache(a["key"], a["value"], a["ks"], a["vs"], a["key_cache"],
                                    a["value_cache"], a["slots"], a["T"], a["Hk"], a["d"], a["bs"],
                                    a["nb"], a["src"], a["kv"], a["k_scale"], a["v_scale"], None)


@pytest.mark.parametrize("over,status", [
    (dict(ks=100), 1),            # token stride shorter than a row
    (dict(d=100), 2),
    (dict(d=120, kv=1), 1),
    (dict(bs=12), 2),
    (dict(src=2), 2),
    (dict(k_scale=0.0, kv=1), 1),
    (dict(key=None), 1),
    (dict(key_cache=0x10004), 1),
    (dict(nb=0), 1),
])
def test_cache_writer_rejects_invalid_arguments_on_host(over, status):
    assert _cache_raw(**over) == status


def test_cache_writer_with_zero_tokens_is_a_noop():
    assert _cache_raw(T=0, key=None) == 0


def test_noalloc_entry_point_host_checks():
    lib = pa.load()
    P = 0x10000
    # 64 x 32 heads x d128 at 64K tokens: ~256 MiB of workspace -> PA_ERR_SCRATCH_TOO_SMALL (4)
    assert lib.pa_v2_decode_noalloc(P, P, P, P, 64, 32, 8, 128, 0.088, P, 4096, 100, P, 16, 65536,
                                    None, 0, 0, 1.0, 1.0, None) == 4
    # a null output is rejected before anything else happens
    assert lib.pa_v2_decode_noalloc(None, P, P, P, 2, 8, 2, 128, 0.088, P, 64, 100, P, 16, 1024,
                                    None, 0, 0, 1.0, 1.0, None) == 1
    assert pa.pa_status_string(4).startswith("step needs more")


def test_block_moves_host_checks():
    lib = pa.load()
    P = 0x10000
    two = (ctypes.c_void_p * 2)(P, P)
    bad = (ctypes.c_void_p * 2)(P, 0x10008)
    assert lib.pa_copy_blocks(two, two, 2, P, 4, 4100, 10, None) == 1   # block bytes not a multiple of 16
    assert lib.pa_copy_blocks(two, bad, 2, P, 4, 4096, 10, None) == 1   # misaligned cache
    assert lib.pa_copy_blocks(two, two, 2, None, 4, 4096, 10, None) == 1
    assert lib.pa_copy_blocks(two, two, 0, P, 4, 4096, 10, None) == 0   # nothing to do
    m = (ctypes.c_int64 * 4)(0, 1, 2, 9)
    assert lib.pa_swap_blocks(P, P, m, 2, 4096, 4, 8, None) == 1        # dst id 9 outside 8 blocks
    m2 = (ctypes.c_int64 * 2)(5, 1)
    assert lib.pa_swap_blocks(P, P, m2, 1, 4096, 4, 8, None) == 1       # src id 5 outside 4 blocks
    assert lib.pa_swap_blocks(P, P, m2, 0, 4096, 4, 8, None) == 0


def _prefix_raw(**over):
    """Call pa_prefix with fake (never dereferenced) pointers; returns the status."""
    lib = pa.load()
    P = 0x10000
    a = dict(output=P, query=P, key=P, value=P, key_cache=P, value_cache=P, num_seqs=2, num_heads=8,
             num_kv_heads=2, head_size=128, scale=0.088, block_tables=P, max_blocks_per_seq=64,
             num_blocks=100, qsl=P, ctx=P, max_query_len=0, block_size=16, q_stride=1024,
             kv_stride=256, dtype=0, ws=None, ws_bytes=0, max_splits=1, split_keys=0)
    a.update(over)
    return lib.pa_prefix(a["output"], a["query"], a["key"], a["value"], a["key_cache"], a["value_cache"],
                         a["num_seqs"], a["num_heads"], a["num_kv_heads"], a["head_size"], a["scale"],
                         a["block_tables"], a["max_blocks_per_seq"], a["num_blocks"], a["qsl"], a["ctx"],
                         a["max_query_len"], a["block_size"], a["q_stride"], a["kv_stride"], a["dtype"], a["ws"],
                         a["ws_bytes"], a["max_splits"], a["split_keys"], None)


@pytest.mark.parametrize("over,status", [
    (dict(num_seqs=-1), 1), (dict(num_heads=6, num_kv_heads=4), 1), (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1), (dict(max_query_len=-1), 1), (dict(head_size=72), 2),
    (dict(block_size=64), 2), (dict(dtype=2), 2), (dict(q_stride=1000), 1), (dict(kv_stride=260), 1),
    (dict(max_blocks_per_seq=0), 1), (dict(max_query_len=5, output=0x10008), 1),
    (dict(max_query_len=5, key=None), 1),
    (dict(num_blocks=1 << 29, num_kv_heads=4, num_heads=8), 1),
])
def test_prefix_rejects_invalid_arguments_on_host(over, status):
    assert _prefix_raw(**over) == status


def test_prefix_with_nothing_to_do_is_a_noop():
    assert _prefix_raw(max_query_len=0) == 0
    assert _prefix_raw(num_seqs=0, max_query_len=9) == 0


def test_prefix_workspace_size():
    lib = pa.load()
    # 2 sequences x 2 kv heads x ceil(100 * 4 / 128) = 4 row tiles x 4 parts x 128 rows x (128 * 4 + 8)
    assert lib.pa_prefix_workspace_size(2, 8, 2, 128, 100, 4) == 2 * 2 * 4 * 4 * 128 * 520
    assert lib.pa_prefix_workspace_size(1, 24, 4, 256, 1024, 6) == 4 * 48 * 6 * 128 * 1032
    assert lib.pa_prefix_workspace_size(2, 8, 2, 128, 100, 1) == 0     # no splitting, no workspace
    assert lib.pa_prefix_workspace_size(2, 8, 2, 128, 100, 33) == 0    # more parts than allowed
    assert lib.pa_prefix_workspace_size(2, 6, 4, 128, 100, 4) == 0     # heads not a multiple
    assert pa.prefix_workspace_size(2, 8, 2, 128, 100, 4) == 2 * 2 * 4 * 4 * 128 * 520


_WS = 2 * 2 * 1 * 4 * 128 * 520  # 2 sequences x 2 kv heads x 1 row tile (5 tokens x 4) x 4 parts


@pytest.mark.parametrize("over", [
    dict(max_splits=33),                              # above the 32-part limit
    dict(split_keys=100),                             # not a multiple of 64
    dict(split_keys=-64),
    dict(ws=0x10008),                                 # workspace not 16-byte aligned
    dict(ws_bytes=_WS - 1),                           # one byte short
])
def test_prefix_rejects_bad_split_workspace(over):
    args = dict(max_query_len=5, ws=0x20000, ws_bytes=_WS, max_splits=4)
    args.update(over)
    assert _prefix_raw(**args) == 1


def test_prefix_ignores_workspace_arguments_when_not_splitting():
    # max_splits <= 1 or no workspace: the split arguments are not looked at
    assert _prefix_raw(max_query_len=0, ws=0x10008, ws_bytes=1, max_splits=1, split_keys=100) == 0
    assert _prefix_raw(max_query_len=0, ws=None, ws_bytes=0, max_splits=8, split_keys=100) == 0


def test_prefix_num_parts_host_plan():
    # no device is touched on these paths: argument checks, no workspace, an explicit split size
    lib = pa.load()
    n = ctypes.c_int(-1)
    F16 = pa.PA_DT_F16
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 1024, 16, 8, 0, 1, None) == 1  # no output
    assert lib.pa_prefix_num_parts(30, 8, 128, F16, 512, 1024, 16, 8, 0, 1, ctypes.byref(n)) == 1  # H % Hk
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 1024, 16, 33, 0, 1, ctypes.byref(n)) == 1  # > 32 parts
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 1024, 16, 8, 100, 1, ctypes.byref(n)) == 1  # % 64
    assert lib.pa_prefix_num_parts(32, 8, 100, F16, 512, 1024, 16, 8, 0, 1, ctypes.byref(n)) == 2  # head size
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 1024, 16, 8, 0, 0, ctypes.byref(n)) == 0 and n.value == 1
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 1024, 16, 1, 0, 1, ctypes.byref(n)) == 0 and n.value == 1
    # 16384-token tables cut at 4096 keys: 4 parts (at most max_splits)
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 1024, 16, 8, 4096, 1, ctypes.byref(n)) == 0 and n.value == 4
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 1024, 16, 3, 4096, 1, ctypes.byref(n)) == 0 and n.value == 3
    # tables no longer than the split size: never cut
    assert lib.pa_prefix_num_parts(32, 8, 128, F16, 512, 256, 16, 8, 4096, 1, ctypes.byref(n)) == 0 and n.value == 1


def test_binding_checks_arguments_before_any_device_call():
    # the ctypes binding rejects what the C ABI cannot take, with CPU tensors, on a machine
    # without a GPU: nothing reaches the library
    import torch
    q = torch.zeros(2, 4, 64, dtype=torch.float16)
    kc = torch.zeros(8, 2, 8, 16, 8, dtype=torch.float16)
    vc = torch.zeros(8, 2, 64, 16, dtype=torch.float16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    sl = torch.ones(2, dtype=torch.int32)
    out = torch.zeros_like(q)
    es = ml = torch.zeros(2, 4, 1)
    tmp = torch.zeros(2, 4, 1, 64)
    # decode: device tensors
    with pytest.raises(ValueError):
        pa.pa_v2_decode(out, es, ml, tmp, q, kc, vc, 2, 0.125, bt, sl, 16, 64)
    # scales: both floats or both per-kv-head float32 CUDA tensors of num_kv_heads values
    assert pa._head_scales(0.5, 0.25, 2) is None
    with pytest.raises(TypeError):
        pa._head_scales(torch.ones(2), 1.0, 2)
    with pytest.raises(TypeError):
        pa._head_scales(torch.ones(2), torch.ones(2), 2)    # CPU tensors
    # block swaps: the mapping is an int64 host tensor [n, 2]
    src = torch.zeros(4, 256, dtype=torch.uint8)
    dst = torch.zeros(4, 256, dtype=torch.uint8)
    with pytest.raises(TypeError):
        pa.pa_swap_blocks(src, dst, torch.zeros(1, 2, dtype=torch.int32))
    with pytest.raises(TypeError):
        pa.pa_swap_blocks(src, dst, torch.zeros(2, dtype=torch.int64))
    with pytest.raises(ValueError):
        pa.pa_swap_blocks(src, torch.zeros(4, 128, dtype=torch.uint8), torch.zeros(1, 2, dtype=torch.int64))
    # prefix: device tensors with dense heads
    with pytest.raises(ValueError):
        pa.pa_prefix(out, q, q[:, :2], q[:, :2], kc, vc, bt, torch.zeros(3, dtype=torch.int32),
                     torch.zeros(2, dtype=torch.int32), 1)
    # the parts query reports the library's own argument checks
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.prefix_num_parts(30, 8, 128, torch.float16, 512, 1024, 16)
    assert e.value.status == 1
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.prefix_num_parts(32, 8, 100, torch.float16, 512, 1024, 16)
    assert e.value.status == 2
    assert pa.prefix_num_parts(32, 8, 128, torch.float16, 512, 1024, 16, 8, 4096) == 4
