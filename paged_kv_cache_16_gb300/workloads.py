"""Seeded synthetic batches shaped like the five workloads of the paged-KV step.

This module only *draws inputs*: request lengths, block tables, random q/k/v
and cache contents, and poison in slots no result may depend on.  It holds
none of the step's arithmetic (no slot computation, no scatter, no
attention); both the CUDA library and the CPU oracle receive exactly the
tensors produced here.

Recipe (all seeded):
  * lengths: ``numpy.random.default_rng(seed).integers(lo, hi + 1)``;
  * physical blocks: one ``rng.permutation(num_blocks)`` of the pool; the
    first id becomes the poison block that pads every block-table row, the
    rest are handed out in request order (shared prefixes take theirs once);
  * q, new key/value and the whole cache pool: N(0, 1) from a seeded
    ``torch.Generator`` (CPU for small pools, the CUDA device for large ones),
    rounded to bfloat16 (round-to-nearest-even);
  * poison: slots past each request's ``seq_len`` inside its last block, the
    slots the step's new tokens will be written to, and the padding block are
    overwritten with a large finite value (3.0e4, alternating sign) or NaN;
  * FP8 (E4M3) caches: the same N(0, 1) pool divided by the tensor's scale and
    cast with torch's float8_e4m3fn conversion (clamped to +-448), so the codes
    spread over the format's range; poison is the code 0x7E (448) or 0x7F (NaN).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16
POISON_FINITE = 30000.0


@dataclass
class Batch:
    name: str
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    num_blocks: int
    query_start_loc: np.ndarray      # int32 [R+1]
    seq_lens: np.ndarray             # int32 [R]
    num_computed: np.ndarray         # int32 [R]
    block_table: np.ndarray          # int32 [R, max_blocks]
    num_common_prefix_blocks: int
    softmax_scale: float
    q: torch.Tensor                  # bf16 [T, Hq, D]
    key: torch.Tensor                # bf16 [T, Hkv, D]  (new tokens)
    value: torch.Tensor              # bf16 [T, Hkv, D]
    key_cache: torch.Tensor          # bf16 [num_blocks, block_size, Hkv, D]
    value_cache: torch.Tensor        # bf16 [num_blocks, block_size, Hkv, D]
    poison_block: int
    meta: dict = field(default_factory=dict)
    kv_cache_dtype: str = "bf16"     # "bf16" or "fp8" (E4M3 codes, uint8 caches)
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def num_reqs(self) -> int:
        return int(len(self.seq_lens))

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc).astype(np.int32)

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_table.shape[1])


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor as a numpy uint16 array of its bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor on ``device``."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) bf16 drawn in chunks so a large pool never needs an fp32 copy."""
    numel = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(numel, dtype=torch.bfloat16, device=device)
    chunk = 1 << 26
    for start in range(0, numel, chunk):
        n = min(chunk, numel - start)
        out[start:start + n] = torch.randn(n, generator=gen, device=device,
                                           dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def _poison_codes(n: int, kind: str, device) -> torch.Tensor:
    """E4M3 poison: the NaN code or the largest finite code, alternating sign."""
    if kind == "nan":
        return torch.full((n,), 0x7F, dtype=torch.uint8, device=device)
    codes = torch.full((n,), 0x7E, dtype=torch.uint8, device=device)
    codes[1::2] = 0xFE
    return codes


def _to_e4m3(pool: torch.Tensor, scale: float) -> torch.Tensor:
    """bf16 pool -> E4M3 codes of pool / scale (torch's cast, clamped)."""
    out = torch.empty(pool.shape, dtype=torch.uint8, device=pool.device)
    flat_in, flat_out = pool.reshape(-1), out.reshape(-1)
    chunk = 1 << 26
    for start in range(0, flat_in.numel(), chunk):
        x = flat_in[start:start + chunk].float() / scale
        flat_out[start:start + chunk] = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def _poison_values(n: int, kind: str, device) -> torch.Tensor:
    if kind == "nan":
        return torch.full((n,), float("nan"), dtype=torch.bfloat16, device=device)
    sign = torch.ones(n, dtype=torch.float32, device=device)
    sign[1::2] = -1.0
    return (sign * POISON_FINITE).to(torch.bfloat16)


def make_batch(*, name: str, num_heads_q: int, num_heads_kv: int, head_dim: int,
               q_lens, seq_lens, num_blocks: int, seed: int = 0,
               shared_prefix: list[tuple[list[int], int]] | None = None,
               num_common_prefix_blocks: int = 0, max_blocks_per_req: int | None = None,
               poison: str = "finite", device="cpu", pool_device=None,
               block_size: int = BLOCK_SIZE, kv_cache_dtype: str = "bf16", k_scale: float = 0.0125,
               v_scale: float = 0.0125) -> Batch:
    """Build one batch.

    q_lens[r] new tokens are scheduled for request r whose total length after
    the step is seq_lens[r]; num_computed = seq_lens - q_lens tokens are
    already in the cache.  ``shared_prefix`` lists (request ids, n_blocks):
    those requests map their first n_blocks logical blocks to the same
    physical blocks.  ``pool_device`` is where the cache pool is drawn
    (default: ``device``).
    """
    q_lens = np.asarray(q_lens, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    assert q_lens.shape == seq_lens.shape
    assert np.all(q_lens >= 0) and np.all(seq_lens >= q_lens)
    R = len(seq_lens)
    num_computed = seq_lens - q_lens
    qsl = np.zeros(R + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(q_lens)
    T = int(qsl[-1])
    n_blocks_req = (seq_lens + block_size - 1) // block_size
    max_blocks = int(max_blocks_per_req or max(1, int(n_blocks_req.max(initial=1))))

    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_blocks)
    poison_block = int(perm[0])
    free = list(perm[1:])
    cursor = 0
    table = np.full((R, max_blocks), poison_block, dtype=np.int64)
    shared_ids: dict[int, np.ndarray] = {}
    for members, n in (shared_prefix or []):
        ids = np.asarray(free[cursor:cursor + n], dtype=np.int64)
        cursor += n
        for r in members:
            assert n_blocks_req[r] >= n
            shared_ids[r] = ids
    for r in range(R):
        start = 0
        if r in shared_ids:
            ids = shared_ids[r]
            table[r, :len(ids)] = ids
            start = len(ids)
        need = int(n_blocks_req[r]) - start
        if need > 0:
            if cursor + need > len(free):
                raise ValueError(f"pool of {num_blocks} blocks too small for {name}")
            table[r, start:start + need] = free[cursor:cursor + need]
            cursor += need

    dev = torch.device(device)
    pdev = torch.device(pool_device) if pool_device is not None else dev
    gen_small = torch.Generator(device=dev).manual_seed(seed * 1000 + 1)
    gen_pool = torch.Generator(device=pdev).manual_seed(seed * 1000 + 2)
    q = _randn_bf16((T, num_heads_q, head_dim), gen_small, dev)
    key = _randn_bf16((T, num_heads_kv, head_dim), gen_small, dev)
    value = _randn_bf16((T, num_heads_kv, head_dim), gen_small, dev)
    kc = _randn_bf16((num_blocks, block_size, num_heads_kv, head_dim), gen_pool, pdev)
    vc = _randn_bf16((num_blocks, block_size, num_heads_kv, head_dim), gen_pool, pdev)

    fp8 = kv_cache_dtype == "fp8"
    if fp8:
        kc, vc = _to_e4m3(kc, k_scale), _to_e4m3(vc, v_scale)
    poison_fn = _poison_codes if fp8 else _poison_values

    # Poison: (a) the padding block, (b) every slot at or past num_computed in
    # a request's own (unshared) blocks -- the new tokens' destinations and
    # the unwritten tail of the last block.
    row = num_heads_kv * head_dim
    kc[poison_block] = poison_fn(block_size * row, poison, pdev).view(block_size, num_heads_kv, head_dim)
    vc[poison_block] = poison_fn(block_size * row, poison, pdev).view(block_size, num_heads_kv, head_dim)
    blocks, offsets = [], []
    for r in range(R):
        first = int(num_computed[r])
        last = int(n_blocks_req[r]) * block_size
        for p in range(first, last):
            blocks.append(table[r, p // block_size])
            offsets.append(p % block_size)
    if blocks:
        b = torch.as_tensor(np.asarray(blocks), device=pdev)
        o = torch.as_tensor(np.asarray(offsets), device=pdev)
        n = len(blocks)
        kc[b, o] = poison_fn(n * row, poison, pdev).view(n, num_heads_kv, head_dim)
        vc[b, o] = poison_fn(n * row, poison, pdev).view(n, num_heads_kv, head_dim)

    return Batch(name=name, num_heads_q=num_heads_q, num_heads_kv=num_heads_kv,
                 head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
                 query_start_loc=qsl.astype(np.int32), seq_lens=seq_lens.astype(np.int32),
                 num_computed=num_computed.astype(np.int32), block_table=table.astype(np.int32),
                 num_common_prefix_blocks=int(num_common_prefix_blocks),
                 softmax_scale=1.0 / math.sqrt(head_dim), q=q, key=key, value=value,
                 key_cache=kc, value_cache=vc, poison_block=poison_block,
                 meta={"seed": seed, "poison": poison}, kv_cache_dtype=kv_cache_dtype,
                 k_scale=float(k_scale) if fp8 else 1.0, v_scale=float(v_scale) if fp8 else 1.0)


# ---------------------------------------------------------------------------
# The five workloads.  Sizes follow the configurations of the step; the
# ``scale`` argument shrinks batch sizes and lengths for CPU-checkable cases.
# ---------------------------------------------------------------------------

def tiny(reading: str = "1A", seed: int = 0, poison: str = "finite", device="cpu") -> Batch:
    """Tiny mixed step: Hq=4, Hkv=2, D=64, 64-block permuted pool, 4 requests.

    The configuration lists contexts 5/17/33/64, two decodes, and prefill
    chunks of 8 and 33 new tokens from num_computed 0, which cannot all hold
    at once.  Reading 1A keeps the new-token counts and num_computed:
    decodes of length 5 and 17, prefills of 8 and 33 from scratch.  Reading
    1B keeps the contexts: decodes of length 5 and 64, a 33-token prefill
    from scratch and an 8-token chunk over a context of 17 (9 computed).
    """
    if reading == "1A":
        q_lens, seq_lens = [1, 1, 8, 33], [5, 17, 8, 33]
    elif reading == "1B":
        q_lens, seq_lens = [1, 1, 8, 33], [5, 64, 17, 33]
    else:
        raise ValueError(reading)
    return make_batch(name=f"tiny-{reading}", num_heads_q=4, num_heads_kv=2, head_dim=64,
                      q_lens=q_lens, seq_lens=seq_lens, num_blocks=64, seed=seed,
                      poison=poison, device=device)


def decode(seed: int = 0, batch: int = 64, lo: int = 512, hi: int = 4096, num_blocks: int = 20000,
           poison: str = "finite", device="cpu", pool_device=None, kv_cache_dtype: str = "bf16") -> Batch:
    """Decode-only Llama-3-8B-shaped layer: Hq=32, Hkv=8, D=128, 64 requests,
    seq_len ~ U[512, 4096] (including the new token), one query token each."""
    rng = np.random.default_rng(seed + 7)
    seq = rng.integers(lo, hi + 1, size=batch)
    return make_batch(name="decode", num_heads_q=32, num_heads_kv=8, head_dim=128,
                      q_lens=np.ones(batch, dtype=np.int64), seq_lens=seq,
                      num_blocks=num_blocks, seed=seed, poison=poison, device=device,
                      pool_device=pool_device, kv_cache_dtype=kv_cache_dtype)


def verify(seed: int = 0, batch: int = 64, q_len: int = 4, lo: int = 512, hi: int = 4096, num_blocks: int = 20000,
           poison: str = "finite", device="cpu", pool_device=None, kv_cache_dtype: str = "bf16") -> Batch:
    """Speculative-decoding verify step on the decode workload's shape: 64
    requests each scoring q_len tokens (the last accepted token + q_len - 1
    drafts) over seq_len ~ U[512, 4096] (including the q_len new tokens)."""
    rng = np.random.default_rng(seed + 11)
    seq = rng.integers(lo, hi + 1, size=batch)
    return make_batch(name="verify", num_heads_q=32, num_heads_kv=8, head_dim=128,
                      q_lens=np.full(batch, q_len, dtype=np.int64), seq_lens=seq,
                      num_blocks=num_blocks, seed=seed, poison=poison, device=device,
                      pool_device=pool_device, kv_cache_dtype=kv_cache_dtype)


def mixed(seed: int = 0, n_decode: int = 256, lo: int = 1024, hi: int = 8192, n_shared: int = 32,
          shared_tokens: int = 1024, chunk: int = 2048, chunk_b_cached: int = 4096,
          poison: str = "finite", device="cpu", pool_device=None, kv_cache_dtype: str = "bf16") -> Batch:
    """Mixed continuous-batching step under an 8192-token budget: 256 decodes
    with seq_len ~ U[1024, 8192], 32 of which share a 1024-token prefix (the
    same 64 physical blocks; their lengths are drawn from [1025, 8192] so the
    new token never lands in a shared block), then a 2048-token chunk from
    scratch and a 2048-token chunk over 4096 cached tokens.  The shared
    prefix covers only part of the batch, so num_common_prefix_blocks = 0."""
    rng = np.random.default_rng(seed + 11)
    seq = rng.integers(lo, hi + 1, size=n_decode)
    members = sorted(rng.choice(n_decode, size=n_shared, replace=False).tolist()) if n_shared else []
    for r in members:
        seq[r] = max(int(seq[r]), shared_tokens + 1)
    q_lens = np.concatenate([np.ones(n_decode, dtype=np.int64), [chunk, chunk]])
    seq_lens = np.concatenate([seq, [chunk, chunk_b_cached + chunk]])
    need = int(((seq_lens + BLOCK_SIZE - 1) // BLOCK_SIZE).sum())
    num_blocks = int(math.ceil((need + 1024) / 1024) * 1024)
    sp = [(members, shared_tokens // BLOCK_SIZE)] if n_shared else None
    return make_batch(name="mixed", num_heads_q=32, num_heads_kv=8, head_dim=128,
                      q_lens=q_lens, seq_lens=seq_lens, num_blocks=num_blocks, seed=seed,
                      shared_prefix=sp, poison=poison, device=device, pool_device=pool_device,
                      kv_cache_dtype=kv_cache_dtype)


def long_context(seed: int = 0, batch: int = 8, context: int = 131072, num_blocks: int = 70000,
                 poison: str = "finite", device="cpu", pool_device=None, kv_cache_dtype: str = "bf16") -> Batch:
    """Long-context decode, 70B-shaped layer: Hq=64, Hkv=8, D=128, 8 requests
    of 131072 tokens each, one query token each, random block permutation."""
    return make_batch(name="long", num_heads_q=64, num_heads_kv=8, head_dim=128,
                      q_lens=np.ones(batch, dtype=np.int64),
                      seq_lens=np.full(batch, context, dtype=np.int64), num_blocks=num_blocks,
                      seed=seed, poison=poison, device=device, pool_device=pool_device,
                      kv_cache_dtype=kv_cache_dtype)


def cascade(seed: int = 0, batch: int = 128, prefix_tokens: int = 4096, lo: int = 64,
            hi: int = 1024, use_cascade: bool = True, num_blocks: int = 8192,
            poison: str = "finite", device="cpu", pool_device=None, kv_cache_dtype: str = "bf16") -> Batch:
    """Cascade shared-prefix decode: 128 decodes over one 4096-token prefix
    (256 shared blocks) plus private suffixes ~ U[64, 1024] (including the new
    token).  ``use_cascade`` sets num_common_prefix_blocks to 256 or 0 on
    otherwise identical inputs."""
    rng = np.random.default_rng(seed + 13)
    suffix = rng.integers(lo, hi + 1, size=batch)
    n_prefix = prefix_tokens // BLOCK_SIZE
    return make_batch(name="cascade" if use_cascade else "cascade-off", num_heads_q=32,
                      num_heads_kv=8, head_dim=128, q_lens=np.ones(batch, dtype=np.int64),
                      seq_lens=prefix_tokens + suffix, num_blocks=num_blocks, seed=seed,
                      shared_prefix=[(list(range(batch)), n_prefix)],
                      num_common_prefix_blocks=n_prefix if use_cascade else 0,
                      poison=poison, device=device, pool_device=pool_device, kv_cache_dtype=kv_cache_dtype)


CONFIGS = {
    "tiny": tiny,
    "decode": decode,
    "mixed": mixed,
    "long": long_context,
    "cascade": cascade,
}
