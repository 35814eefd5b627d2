"""Seeded synthetic inputs for paged single-query decode attention.

This module only builds data: shapes, value distributions, block-table permutations,
sequence-length mixes and NaN canaries.  It holds none of the attention arithmetic, so
the CPU oracle and the CUDA path can both consume the bytes it produces without sharing
any of the method's code.

Layouts follow "paged_attention_v2_pytorch.py" (argument comments of
``paged_attention_v2_pytorch``) and "paged_attn.py" (``split_kv_cache``):

* ``query``       [num_seqs, num_heads, head_size]
* ``key_cache``   [num_blocks, num_kv_heads, head_size // x, block_size, x], x = 16 / elem bytes
* ``value_cache`` [num_blocks, num_kv_heads, head_size, block_size]
* ``block_tables`` int32 [num_seqs, max_blocks_per_seq], ``seq_lens`` int32 [num_seqs]

Element storage: fp16 and bf16 tensors as themselves; the fp8 e4m3 cache as a uint8
tensor of codes (quantised with torch's own ``float8_e4m3fn`` cast of ``x / k_scale``).

Canaries: every physical block no sequence uses, every table entry past a sequence's
last block, and every slot past ``seq_len`` in a sequence's last block hold NaN, so a
read of a masked slot that reaches a result shows up as NaN instead of passing silently.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np
import torch

PARTITION_SIZE = 512  # tokens per partition ("paged_attention_v2_pytorch.py", _PARTITION_SIZE)

# NaN bit patterns per storage format.
_NAN_CODE = {"f16": 0x7E00, "bf16": 0x7FC0, "fp8_e4m3": 0x7F}

_CHUNK = 1 << 22  # elements per independently seeded RNG chunk


@dataclasses.dataclass
class Workload:
    """One decode step's inputs, all on the host (torch CPU tensors)."""

    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    q_dtype: str  # "f16" | "bf16"
    kv_cache_dtype: str  # "auto" (same as q) | "fp8_e4m3"
    scale: float
    k_scale: float
    v_scale: float
    query: torch.Tensor  # [S, H, d] q dtype
    key_cache: torch.Tensor  # [NB, Hk, d/x, bs, x] q dtype, or uint8 codes
    value_cache: torch.Tensor  # [NB, Hk, d, bs]
    block_tables: torch.Tensor  # int32 [S, max_blocks_per_seq]
    seq_lens: torch.Tensor  # int32 [S]
    alibi_slopes: Optional[torch.Tensor]  # float32 [H] or None
    max_seq_len: int
    # The cache writer's inputs for this step: the newest token of every sequence.
    new_key: torch.Tensor  # [S, Hk, d] q dtype
    new_value: torch.Tensor  # [S, Hk, d] q dtype
    slot_mapping: torch.Tensor  # int64 [S]; -1 for empty sequences
    sigma: float = 1.0
    seed: int = 0
    # One scale per kv head (float32 [Hk]) in place of k_scale / v_scale, or None.
    k_scales: Optional[torch.Tensor] = None
    v_scales: Optional[torch.Tensor] = None

    def k_scales_or_scalar(self):
        return self.k_scale if self.k_scales is None else self.k_scales

    def v_scales_or_scalar(self):
        return self.v_scale if self.v_scales is None else self.v_scales

    @property
    def x(self) -> int:
        return 16 // self.kv_elem_bytes

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_cache_dtype == "fp8_e4m3" else 2

    @property
    def q_elem_bytes(self) -> int:
        return 2

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_num_partitions(self) -> int:
        return max(1, -(-self.max_seq_len // PARTITION_SIZE))

    @property
    def kv_storage(self) -> str:
        return "fp8_e4m3" if self.kv_cache_dtype == "fp8_e4m3" else self.q_dtype

    def algorithmic_bytes(self) -> int:
        """Bytes one decode step must move: every valid K and V element once per kv-head,
        plus the query read and the output write (workspace excluded)."""
        toks = int(self.seq_lens.to(torch.int64).sum())
        kv = toks * self.num_kv_heads * self.head_size * self.kv_elem_bytes * 2
        q = self.num_seqs * self.num_heads * self.head_size * self.q_elem_bytes
        return kv + 2 * q

    def writer_bytes(self) -> int:
        """Bytes of the cache-write step: read new K/V rows and the slot map, write the slots."""
        n = int((self.slot_mapping >= 0).sum())
        row = self.num_kv_heads * self.head_size
        return n * row * (self.q_elem_bytes + self.kv_elem_bytes) * 2 + self.num_seqs * 8


# --------------------------------------------------------------------------------------
# Named workloads: the five decode configurations this library is measured on, a small
# batch and a 16:1 GQA batch.
# --------------------------------------------------------------------------------------
CONFIGS = {
    "tiny": dict(
        num_seqs=2, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
        lens=("fixed", [37, 600]), num_blocks=64, q_dtype="f16", kv_cache_dtype="auto",
        sigma=1.0, alibi=False, seed=1001,
    ),
    "llama_gqa_decode": dict(
        num_seqs=64, num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
        lens=("uniform", 1, 4096), q_dtype="f16", kv_cache_dtype="auto",
        sigma=1.0, alibi=False, seed=1002,
    ),
    "long_context_gqa": dict(
        num_seqs=4, num_heads=24, num_kv_heads=4, head_size=256, block_size=16,
        lens=("fixed", [100000] * 4), q_dtype="f16", kv_cache_dtype="auto",
        sigma=0.5, alibi=False, seed=1003,
    ),
    "fp8_kv": dict(
        num_seqs=128, num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
        lens=("uniform", 512, 8192), q_dtype="f16", kv_cache_dtype="fp8_e4m3",
        k_scale=0.05, v_scale=0.05, sigma=1.0, alibi=False, seed=1004,
    ),
    "mha_alibi_ragged": dict(
        num_seqs=256, num_heads=16, num_kv_heads=16, head_size=96, block_size=32,
        lens=("lognormal", 1024.0, 1.0, 32768, {0: 0, 1: 1}), q_dtype="bf16",
        kv_cache_dtype="auto", sigma=1.0, alibi=True, seed=1005,
    ),
    # A small batch: two Llama-style sequences of 4K-8K tokens.  Its grid has fewer 512-token
    # units (kv heads x partitions) than the GPU has CTA slots.
    "small_batch_gqa": dict(
        num_seqs=2, num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
        lens=("uniform", 4096, 8192), q_dtype="f16", kv_cache_dtype="auto",
        sigma=1.0, alibi=False, seed=1006,
    ),
    # 8 query heads per kv head (the 64-query / 8-kv-head shape of the larger Llama-style
    # models): a full MMA tile of heads a CTA.
    "gqa8_decode": dict(
        num_seqs=64, num_heads=64, num_kv_heads=8, head_size=128, block_size=16,
        lens=("uniform", 1, 4096), q_dtype="f16", kv_cache_dtype="auto",
        sigma=1.0, alibi=False, seed=1008,
    ),
    # 16 query heads per kv head: more than one MMA tile of heads shares each kv head.
    "gqa16_decode": dict(
        num_seqs=64, num_heads=64, num_kv_heads=4, head_size=128, block_size=16,
        lens=("uniform", 1, 4096), q_dtype="f16", kv_cache_dtype="auto",
        sigma=1.0, alibi=False, seed=1007,
    ),
}

# Reduced-size stand-ins the oracle finishes in seconds: same heads, head size, block
# size, dtypes and length mix, fewer sequences and shorter contexts (still several
# partitions and a ragged tail).
REDUCED = {
    "tiny": {},
    "llama_gqa_decode": dict(num_seqs=6, lens=("uniform", 1, 1600)),
    "long_context_gqa": dict(num_seqs=2, lens=("fixed", [3000, 2561])),
    "fp8_kv": dict(num_seqs=6, lens=("uniform", 512, 1800)),
    "mha_alibi_ragged": dict(num_seqs=8, lens=("lognormal", 300.0, 1.0, 2000, {0: 0, 1: 1})),
    "small_batch_gqa": dict(lens=("uniform", 1200, 2600)),
    "gqa8_decode": dict(num_seqs=4, lens=("uniform", 1, 1600)),
    "gqa16_decode": dict(num_seqs=4, lens=("uniform", 1, 1600)),
}


def alibi_slopes_for(num_heads: int) -> np.ndarray:
    """Slopes 2^(-8(i+1)/H) for head i (the geometric ALiBi schedule)."""
    return np.array([2.0 ** (-8.0 * (i + 1) / num_heads) for i in range(num_heads)],
                    dtype=np.float32)


def _draw_lens(spec, num_seqs: int, rng: np.random.Generator) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        vals = list(spec[1])
        assert len(vals) == num_seqs or num_seqs <= len(vals)
        return np.array(vals[:num_seqs], dtype=np.int64)
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return rng.integers(lo, hi + 1, size=num_seqs, dtype=np.int64)
    if kind == "lognormal":
        median, sig, cap, forced = spec[1], spec[2], spec[3], spec[4]
        v = np.rint(rng.lognormal(mean=math.log(median), sigma=sig, size=num_seqs))
        v = np.clip(v, 1, cap).astype(np.int64)
        for i, L in forced.items():
            if i < num_seqs:
                v[i] = L
        return v
    raise ValueError(f"unknown length spec {spec!r}")


def _fill_normal(shape, sigma: float, seed: int, stream: int) -> np.ndarray:
    """float32 N(0, sigma^2) of the given shape, generated in fixed-size chunks that are
    each seeded from (seed, stream, chunk index), so the result does not depend on the
    number of threads used."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nchunks = -(-n // _CHUNK)

    def work(ci: int) -> None:
        lo = ci * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.default_rng(np.random.SeedSequence([seed, stream, ci]))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if sigma != 1.0:
            out[lo:hi] *= np.float32(sigma)

    threads = min(nchunks, max(1, len(os.sched_getaffinity(0))))
    if threads <= 1:
        for ci in range(nchunks):
            work(ci)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def _to_storage(a: np.ndarray, storage: str, inv_scale=1.0) -> torch.Tensor:
    t = torch.from_numpy(a)
    if storage == "f16":
        return t.to(torch.float16)
    if storage == "bf16":
        return t.to(torch.bfloat16)
    if storage == "fp8_e4m3":
        if isinstance(inv_scale, np.ndarray):  # one scale per kv head, broadcast
            t = t * torch.from_numpy(inv_scale).to(t.dtype)
        elif inv_scale != 1.0:
            t = t * inv_scale
        return t.to(torch.float8_e4m3fn).view(torch.uint8)
    raise ValueError(storage)


def _torch_dtype(name: str) -> torch.dtype:
    return {"f16": torch.float16, "bf16": torch.bfloat16}[name]


def _nan_fill_(t: torch.Tensor, storage: str) -> None:
    code = _NAN_CODE[storage]
    if storage == "fp8_e4m3":
        t.fill_(code)
    else:
        t.view(torch.int16).fill_(code if code < 0x8000 else code - 0x10000)


def build(
    *,
    name: str = "custom",
    num_seqs: int,
    num_heads: int,
    num_kv_heads: int,
    head_size: int,
    block_size: int,
    seq_lens: Sequence[int],
    q_dtype: str = "f16",
    kv_cache_dtype: str = "auto",
    sigma: float = 1.0,
    alibi: bool = False,
    k_scale: float = 1.0,
    v_scale: float = 1.0,
    k_scales: Optional[Sequence[float]] = None,
    v_scales: Optional[Sequence[float]] = None,
    scale: Optional[float] = None,
    num_blocks: Optional[int] = None,
    block_slack: float = 1.25,
    max_seq_len: Optional[int] = None,
    table_width: Optional[int] = None,
    canaries: bool = True,
    seed: int = 0,
) -> Workload:
    """Build one seeded workload.

    Physical block ids come from one ``permutation(num_blocks)`` dealt out sequence by
    sequence; the first unused id is the canary block every padding entry points at.
    ``k_scales`` / ``v_scales`` (num_kv_heads values each) replace k_scale / v_scale per kv
    head: an fp8 cache then holds head j's values quantised as x / k_scales[j].
    """
    rng = np.random.default_rng(seed)
    S, H, Hk, d, bs = num_seqs, num_heads, num_kv_heads, head_size, block_size
    lens = np.asarray(seq_lens, dtype=np.int64)
    assert lens.shape == (S,)
    storage = "fp8_e4m3" if kv_cache_dtype == "fp8_e4m3" else q_dtype
    x = 16 // (1 if storage == "fp8_e4m3" else 2)
    assert d % x == 0, "head_size must be a multiple of x"

    need = [-(-int(L) // bs) for L in lens]
    total = sum(need)
    if num_blocks is None:
        num_blocks = max(total + 1, int(math.ceil(total * block_slack)))
    assert num_blocks > total, "need at least one spare block for the canary"
    msl = int(lens.max()) if max_seq_len is None else int(max_seq_len)
    width = max(1, -(-msl // bs)) if table_width is None else int(table_width)
    assert width >= max(need + [1])

    perm = rng.permutation(num_blocks).astype(np.int64)
    tables = np.empty((S, width), dtype=np.int64)
    spare = perm[total:]
    canary = int(spare[0])
    pos = 0
    for s in range(S):
        n = need[s]
        tables[s, :n] = perm[pos:pos + n]
        tables[s, n:] = canary
        pos += n

    # Values: K and V caches over all physical blocks, then the query and new-token rows.
    kshape = (num_blocks, Hk, d // x, bs, x)
    vshape = (num_blocks, Hk, d, bs)
    ksv = None if k_scales is None else np.asarray(k_scales, dtype=np.float32).reshape(Hk)
    vsv = None if v_scales is None else np.asarray(v_scales, dtype=np.float32).reshape(Hk)
    inv = 1.0 / k_scale if storage == "fp8_e4m3" else 1.0
    if ksv is not None and storage == "fp8_e4m3":
        inv = (1.0 / ksv).astype(np.float32).reshape(1, Hk, 1, 1, 1)
    key_cache = _to_storage(_fill_normal(kshape, sigma, seed, 1), storage, inv)
    inv = 1.0 / v_scale if storage == "fp8_e4m3" else 1.0
    if vsv is not None and storage == "fp8_e4m3":
        inv = (1.0 / vsv).astype(np.float32).reshape(1, Hk, 1, 1)
    value_cache = _to_storage(_fill_normal(vshape, sigma, seed, 2), storage, inv)
    query = _to_storage(_fill_normal((S, H, d), sigma, seed, 3), q_dtype)
    new_key = _to_storage(_fill_normal((S, Hk, d), sigma, seed, 4), q_dtype)
    new_value = _to_storage(_fill_normal((S, Hk, d), sigma, seed, 5), q_dtype)

    if canaries:
        used = np.zeros(num_blocks, dtype=bool)
        used[perm[:total]] = True
        unused = torch.from_numpy(np.nonzero(~used)[0])
        kc = key_cache.index_select(0, unused)
        _nan_fill_(kc, storage)
        key_cache.index_copy_(0, unused, kc)
        vc = value_cache.index_select(0, unused)
        _nan_fill_(vc, storage)
        value_cache.index_copy_(0, unused, vc)
        for s in range(S):
            L = int(lens[s])
            if L > 0 and L % bs:
                b = int(tables[s, need[s] - 1])
                _nan_fill_(key_cache[b, :, :, L % bs:, :], storage)
                _nan_fill_(value_cache[b, :, :, L % bs:], storage)

    slots = np.full(S, -1, dtype=np.int64)
    for s in range(S):
        L = int(lens[s])
        if L > 0:
            t = L - 1
            slots[s] = tables[s, t // bs] * bs + t % bs

    slopes = torch.from_numpy(alibi_slopes_for(H)) if alibi else None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Workload(
        name=name, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=d, block_size=bs,
        num_blocks=num_blocks, q_dtype=q_dtype, kv_cache_dtype=kv_cache_dtype,
        scale=float(np.float32(scale)), k_scale=float(np.float32(k_scale)),
        v_scale=float(np.float32(v_scale)), query=query, key_cache=key_cache,
        value_cache=value_cache, block_tables=torch.from_numpy(tables.astype(np.int32)),
        seq_lens=torch.from_numpy(lens.astype(np.int32)), alibi_slopes=slopes,
        max_seq_len=msl, new_key=new_key, new_value=new_value,
        slot_mapping=torch.from_numpy(slots), sigma=sigma, seed=seed,
        k_scales=None if ksv is None else torch.from_numpy(ksv.copy()),
        v_scales=None if vsv is None else torch.from_numpy(vsv.copy()),
    )


def make(name: str, *, reduced: bool = False, canaries: bool = True,
         seed: Optional[int] = None, **overrides) -> Workload:
    """One of the named workloads (``CONFIGS``), full size or reduced (``REDUCED``)."""
    cfg = dict(CONFIGS[name])
    if reduced:
        cfg.update(REDUCED[name])
    cfg.update(overrides)
    if seed is not None:
        cfg["seed"] = seed
    rng = np.random.default_rng(cfg["seed"] + 7)
    lens = _draw_lens(cfg.pop("lens"), cfg["num_seqs"], rng)
    num_blocks = cfg.pop("num_blocks", None)
    return build(name=name, seq_lens=lens, num_blocks=num_blocks, canaries=canaries, **cfg)


def shard(wl_name: str, rank: int, world: int, **kw) -> Workload:
    """The workload a rank of a multi-GPU run processes: the same configuration drawn with
    a rank-specific seed.  Sequences are independent, so ranks share nothing."""
    base = CONFIGS[wl_name]["seed"]
    return make(wl_name, seed=base + 100_003 * rank, **kw)


# --------------------------------------------------------------------------------------
# Chunked-prefix (prefill) inputs: "paged_attn.py", _forward_prefix_pytorch.
# --------------------------------------------------------------------------------------
@dataclasses.dataclass
class PrefixWorkload:
    """One chunked-prefill step: sequence s has ``context_lens[s]`` tokens already in the
    paged cache and ``q_len = query_start_loc[s+1] - query_start_loc[s]`` new tokens whose
    query/key/value rows are dense.  The block table covers context + new tokens (as a
    serving engine's table would after writing the chunk), but the cache slots of the new
    tokens hold NaN canaries: the method reads the chunk's keys and values from the dense
    ``key``/``value`` rows, never from the cache."""

    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    q_dtype: str
    scale: float
    query: torch.Tensor  # [T, H, d]
    key: torch.Tensor  # [T, Hk, d]
    value: torch.Tensor  # [T, Hk, d]
    key_cache: torch.Tensor  # [NB, Hk, d/x, bs, x]
    value_cache: torch.Tensor  # [NB, Hk, d, bs]
    block_tables: torch.Tensor  # int32 [S, W]
    query_start_loc: torch.Tensor  # int32 [S + 1]
    context_lens: torch.Tensor  # int32 [S]
    seq_lens: torch.Tensor  # int32 [S] context + new tokens
    max_query_len: int
    seed: int = 0

    @property
    def x(self) -> int:
        return 8

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def query_lens(self) -> np.ndarray:
        q = self.query_start_loc.numpy().astype(np.int64)
        return q[1:] - q[:-1]

    def flops(self) -> int:
        """Multiply-adds x 2 of the two products: query token j of a sequence with context c
        sees c + j + 1 keys, each costing d MACs for the score and d for the value sum."""
        c = self.context_lens.numpy().astype(np.int64)
        q = self.query_lens
        keys = (q * c + q * (q + 1) // 2).sum()
        return int(4 * self.head_size * self.num_heads * keys)

    def algorithmic_bytes(self) -> int:
        """Bytes read and written once: context K/V per kv head, the chunk's q/k/v rows, out."""
        c = int(self.context_lens.to(torch.int64).sum())
        T, H, Hk, d = self.num_tokens, self.num_heads, self.num_kv_heads, self.head_size
        return 2 * (2 * c * Hk * d + T * (2 * H + 2 * Hk) * d)


PREFIX_CONFIGS = {
    "prefix_tiny": dict(
        num_seqs=3, num_heads=4, num_kv_heads=2, head_size=64, block_size=16,
        context_lens=[0, 37, 600], query_lens=[5, 70, 129], q_dtype="f16", seed=2001,
    ),
    # The pages' model shape (24 query heads, 4 kv heads, head size 256) with one chunked
    # prefill step of 4096 new tokens (the pages' max_num_batched_tokens) split over four
    # sequences whose cached prefixes run from none to ~100K tokens.
    "prefix_long_gqa": dict(
        num_seqs=4, num_heads=24, num_kv_heads=4, head_size=256, block_size=16,
        context_lens=[0, 8192, 32768, 98304], query_lens=[1024] * 4, q_dtype="f16",
        sigma=0.5, seed=2002,
    ),
    # Llama-style GQA (32/8, d 128): eight sequences of 512 new tokens over cached prefixes
    # drawn uniformly from [0, 16384].
    "prefix_llama_gqa": dict(
        num_seqs=8, num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
        context_lens=("uniform", 0, 16384), query_lens=[512] * 8, q_dtype="bf16", seed=2003,
    ),
}

PREFIX_REDUCED = {
    "prefix_tiny": {},
    "prefix_long_gqa": dict(num_seqs=3, context_lens=[0, 700, 1500], query_lens=[200, 131, 64]),
    "prefix_llama_gqa": dict(num_seqs=4, context_lens=("uniform", 0, 900),
                             query_lens=[100, 1, 257, 64]),
}


def build_prefix(*, name: str = "custom", num_seqs: int, num_heads: int, num_kv_heads: int,
                 head_size: int, block_size: int, context_lens: Sequence[int],
                 query_lens: Sequence[int], q_dtype: str = "f16", sigma: float = 1.0,
                 scale: Optional[float] = None, block_slack: float = 1.25,
                 table_width: Optional[int] = None, canaries: bool = True,
                 seed: int = 0) -> PrefixWorkload:
    """Seeded chunked-prefill inputs; block ids dealt from one permutation as in ``build``."""
    rng = np.random.default_rng(seed)
    S, H, Hk, d, bs = num_seqs, num_heads, num_kv_heads, head_size, block_size
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    assert ctx.shape == (S,) and ql.shape == (S,) and d % 8 == 0
    tot = ctx + ql
    need = [-(-int(L) // bs) for L in tot]
    total = sum(need)
    num_blocks = max(total + 1, int(math.ceil(total * block_slack)))
    width = max(1, max(need)) if table_width is None else int(table_width)
    assert width >= max(need + [1])
    perm = rng.permutation(num_blocks).astype(np.int64)
    tables = np.empty((S, width), dtype=np.int64)
    canary = int(perm[total])
    pos = 0
    for s in range(S):
        tables[s, :need[s]] = perm[pos:pos + need[s]]
        tables[s, need[s]:] = canary
        pos += need[s]
    T = int(ql.sum())
    key_cache = _to_storage(_fill_normal((num_blocks, Hk, d // 8, bs, 8), sigma, seed, 11), q_dtype)
    value_cache = _to_storage(_fill_normal((num_blocks, Hk, d, bs), sigma, seed, 12), q_dtype)
    query = _to_storage(_fill_normal((T, H, d), sigma, seed, 13), q_dtype)
    key = _to_storage(_fill_normal((T, Hk, d), sigma, seed, 14), q_dtype)
    value = _to_storage(_fill_normal((T, Hk, d), sigma, seed, 15), q_dtype)
    if canaries:
        used = np.zeros(num_blocks, dtype=bool)
        used[perm[:total]] = True
        for b in np.nonzero(~used)[0]:
            _nan_fill_(key_cache[int(b)], q_dtype)
            _nan_fill_(value_cache[int(b)], q_dtype)
        for s in range(S):
            # every slot from the first new token on: the chunk is read from key/value
            for t in range(int(ctx[s]), need[s] * bs):
                b, o = int(tables[s, t // bs]), t % bs
                _nan_fill_(key_cache[b, :, :, o, :], q_dtype)
                _nan_fill_(value_cache[b, :, :, o], q_dtype)
    qsl = np.zeros(S + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(ql)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return PrefixWorkload(
        name=name, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_size=d, block_size=bs,
        num_blocks=num_blocks, q_dtype=q_dtype, scale=float(np.float32(scale)), query=query,
        key=key, value=value, key_cache=key_cache, value_cache=value_cache,
        block_tables=torch.from_numpy(tables.astype(np.int32)),
        query_start_loc=torch.from_numpy(qsl.astype(np.int32)),
        context_lens=torch.from_numpy(ctx.astype(np.int32)),
        seq_lens=torch.from_numpy(tot.astype(np.int32)), max_query_len=int(ql.max(initial=0)),
        seed=seed,
    )


def make_prefix(name: str, *, reduced: bool = False, seed: Optional[int] = None,
                **overrides) -> PrefixWorkload:
    """One of the named chunked-prefill workloads, full size or reduced."""
    cfg = dict(PREFIX_CONFIGS[name])
    if reduced:
        cfg.update(PREFIX_REDUCED[name])
    cfg.update(overrides)
    if seed is not None:
        cfg["seed"] = seed
    c = cfg["context_lens"]
    if isinstance(c, tuple):
        rng = np.random.default_rng(cfg["seed"] + 7)
        cfg["context_lens"] = _draw_lens(c, cfg["num_seqs"], rng)
    return build_prefix(name=name, **cfg)
