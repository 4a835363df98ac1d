"""Seeded synthetic workloads for paged KV-cache attention.

This module is shared by the tests, the bench and the smoke check, and by
both sides of every parity comparison.  It holds inputs only: shapes,
sequence lengths, random physical placement of blocks, and random bf16
values.  It computes no attention, no slot or address mapping and no
copy-on-write plan; those belong to the product and to the oracle, each on
its own.

The shapes follow the pages' worked example, how-pagedattention-works
(aiinfrainterviews.com), "A strong answer": a Llama 3.1 70B layer (64 query
heads, 8 KV heads, head_dim 128, bf16, 16-token blocks), chats of a 600-token
prompt plus up to 250 generated tokens, an 8,192-token maximum, and a
2,000-token shared system prompt; beam forks follow
attn-paged-attention-mcq-hard (zenaique.com), the interviewer follow-up on
beam search.  The page example with 4-slot blocks and table [5, 1, 7] follows
auto-20261007-1900-en (lihaoran.work), "A block table maps logical order to
physical storage".

Values are bf16 drawn from N(0, 1); every generator is seeded (numpy
``default_rng`` for lengths and placement, ``torch.Generator`` for values).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

SEED_BASE = 167


@dataclass
class Workload:
    """Host-side description of one synthetic batch (numpy metadata)."""
    name: str
    kind: str                      # "decode" or "prefill"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    seq_lens: np.ndarray           # int32 [B]: tokens attended by decode (incl. the new one)
    tables: np.ndarray             # int32 [B][max_blocks], -1 where unused
    referenced: np.ndarray         # int64 [n]: physical blocks that hold data
    seed: int
    new_seq_idx: Optional[np.ndarray] = None    # int32 [N]: sequence of each new token
    new_positions: Optional[np.ndarray] = None  # int64 [N]: logical position of each new token
    copy_pairs: Optional[np.ndarray] = None     # int32 [n][2] (src, dst) block forks
    ctx_lens: Optional[np.ndarray] = None       # int32 [B]: prefill cached context
    chunk: int = 0                              # prefill query chunk length
    partition_tokens: int = 0                   # 0 = let the library choose
    notes: Dict[str, object] = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.tables.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        if self.kind == "prefill":
            return int((self.ctx_lens + self.chunk).max())
        return int(self.seq_lens.max()) if self.seq_lens.size else 0


def _blocks_for(tokens: int, block_size: int) -> int:
    # table width needed to hold `tokens` positions (a size, used to shape arrays)
    return -(-tokens // block_size)


def _tables_from_counts(counts: List[int], placement: np.ndarray) -> np.ndarray:
    width = max(1, max(counts) if counts else 1)
    tables = np.full((len(counts), width), -1, dtype=np.int32)
    cursor = 0
    for s, n in enumerate(counts):
        tables[s, :n] = placement[cursor:cursor + n]
        cursor += n
    return tables


def _referenced(tables: np.ndarray, extra=()) -> np.ndarray:
    ids = tables[tables >= 0].astype(np.int64)
    if len(extra):
        ids = np.concatenate([ids, np.asarray(extra, dtype=np.int64)])
    return np.unique(ids)


# ---------------------------------------------------------------------------
# configurations
# ---------------------------------------------------------------------------

def tiny(seed: int = SEED_BASE + 0) -> Workload:
    """4 sequences of {1, 10, 16, 37} tokens, 4/2 heads, d=64, b=16, 32-block
    pool, tables drawn without repetition."""
    rng = np.random.default_rng(seed)
    b, lens = 16, [1, 10, 16, 37]
    counts = [_blocks_for(L, b) for L in lens]
    placement = rng.permutation(32).astype(np.int32)
    tables = _tables_from_counts(counts, placement)
    seq = np.asarray(lens, dtype=np.int32)
    return Workload("tiny", "decode", 4, 2, 64, b, 32, 1.0 / math.sqrt(64), seq, tables,
                    _referenced(tables), seed,
                    new_seq_idx=np.arange(4, dtype=np.int32),
                    new_positions=(seq.astype(np.int64) - 1))


def tiny_page_example(seed: int = SEED_BASE + 0) -> Workload:
    """The page example: 4-slot blocks, one sequence of 10 tokens with table
    [5, 1, 7] in an 8-block pool; 4/2 heads, d=64."""
    tables = np.asarray([[5, 1, 7]], dtype=np.int32)
    seq = np.asarray([10], dtype=np.int32)
    return Workload("tiny_page_example", "decode", 4, 2, 64, 4, 8, 1.0 / math.sqrt(64), seq,
                    tables, _referenced(tables), seed,
                    new_seq_idx=np.arange(10, dtype=np.int32) * 0,
                    new_positions=np.arange(10, dtype=np.int64))


def llama70b_decode(seed: int = SEED_BASE + 1, batch: int = 64) -> Workload:
    """Llama-3.1-70B-shaped single-layer decode: 64/8 heads, d=128, b=16,
    seq_lens uniform in [600, 850] (prompt 600 plus up to 250 generated), blocks
    placed by a random permutation of a 16,384-block pool; the newest token of
    each sequence is written by the slot writer, then attended."""
    rng = np.random.default_rng(seed)
    b, nb = 16, 16384
    lens = rng.integers(600, 851, size=batch).astype(np.int32)
    counts = [_blocks_for(int(L), b) for L in lens]
    tables = _tables_from_counts(counts, rng.permutation(nb).astype(np.int32))
    return Workload("llama70b_decode", "decode", 64, 8, 128, b, nb, 1.0 / math.sqrt(128), lens,
                    tables, _referenced(tables), seed,
                    new_seq_idx=np.arange(batch, dtype=np.int32),
                    new_positions=lens.astype(np.int64) - 1)


def long_context(seed: int = SEED_BASE + 2, batch: int = 8, seq_len: int = 8192) -> Workload:
    """8 sequences of 8,192 tokens (512 blocks each), 64/8 heads, d=128, b=16,
    random placement in an 8,192-block pool, 512-token context partitions."""
    rng = np.random.default_rng(seed)
    b, nb = 16, 8192
    lens = np.full(batch, seq_len, dtype=np.int32)
    counts = [_blocks_for(int(L), b) for L in lens]
    tables = _tables_from_counts(counts, rng.permutation(nb).astype(np.int32))
    return Workload("long_context", "decode", 64, 8, 128, b, nb, 1.0 / math.sqrt(128), lens,
                    tables, _referenced(tables), seed,
                    new_seq_idx=np.arange(batch, dtype=np.int32),
                    new_positions=lens.astype(np.int64) - 1, partition_tokens=512)


def shared_prefix(seed: int = SEED_BASE + 3, batch: int = 256, sigma: float = 0.8) -> Workload:
    """256 sequences sharing one 2,000-token system prompt (125 blocks, the
    same physical ids at the head of every table) followed by private
    suffixes of lognormal length (median 850, sigma 0.8, clipped to
    [1, 6192]); 64/8 heads, d=128, b=16, 32,768-block pool."""
    rng = np.random.default_rng(seed)
    b, nb, prefix_tokens = 16, 32768, 2000
    prefix_blocks = prefix_tokens // b
    suffix = np.clip(np.rint(rng.lognormal(math.log(850.0), sigma, size=batch)), 1, 6192)
    lens = (prefix_tokens + suffix).astype(np.int32)
    placement = rng.permutation(nb).astype(np.int32)
    shared = placement[:prefix_blocks]
    rest = placement[prefix_blocks:]
    width = max(_blocks_for(int(L), b) for L in lens)
    tables = np.full((batch, width), -1, dtype=np.int32)
    cursor = 0
    for s, L in enumerate(lens):
        n_private = _blocks_for(int(L), b) - prefix_blocks
        tables[s, :prefix_blocks] = shared
        tables[s, prefix_blocks:prefix_blocks + n_private] = rest[cursor:cursor + n_private]
        cursor += n_private
    return Workload("shared_prefix", "decode", 64, 8, 128, b, nb, 1.0 / math.sqrt(128), lens,
                    tables, _referenced(tables), seed,
                    new_seq_idx=np.arange(batch, dtype=np.int32),
                    new_positions=lens.astype(np.int64) - 1,
                    notes={"prefix_blocks": prefix_blocks, "shared_ids": shared.copy()})


def beam_fork(seed: int = SEED_BASE + 4, prompts: int = 32, beams: int = 4) -> Workload:
    """32 prompts x 4 beams.  Prompt lengths are uniform in [1024, 3000]; the
    beams of a prompt share its blocks.  When the prompt's last block is only
    partly filled, beam 0 keeps it and beams 1..3 each receive a private copy
    (a (src, dst) fork pair); each beam then appends its own token at position
    Lp and decode attends Lp + 1 tokens (batch 128)."""
    rng = np.random.default_rng(seed)
    b, nb = 16, 8192
    plen = rng.integers(1024, 3001, size=prompts).astype(np.int64)
    placement = iter(rng.permutation(nb).astype(np.int32).tolist())
    B = prompts * beams
    lens = np.repeat(plen + 1, beams).astype(np.int32)
    width = max(_blocks_for(int(L), b) for L in lens)
    tables = np.full((B, width), -1, dtype=np.int32)
    pairs = []
    for p in range(prompts):
        n_prompt = _blocks_for(int(plen[p]), b)
        prompt_ids = [next(placement) for _ in range(n_prompt)]
        partial_tail = int(plen[p]) % b != 0
        for beam in range(beams):
            row = p * beams + beam
            ids = list(prompt_ids)
            if partial_tail:
                if beam > 0:
                    fresh = next(placement)
                    pairs.append((prompt_ids[-1], fresh))
                    ids[-1] = fresh
            else:
                ids.append(next(placement))
            tables[row, :len(ids)] = ids
    copy_pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
    return Workload("beam_fork", "decode", 64, 8, 128, b, nb, 1.0 / math.sqrt(128), lens, tables,
                    _referenced(tables, copy_pairs.ravel()), seed,
                    new_seq_idx=np.arange(B, dtype=np.int32),
                    new_positions=lens.astype(np.int64) - 1, copy_pairs=copy_pairs,
                    notes={"prompt_lens": plen, "beams": beams})


def prefill_chunk(seed: int = SEED_BASE + 4, batch: int = 16, ctx=4096, chunk: int = 512,
                  num_blocks: int = 8192, num_q_heads: int = 64, num_kv_heads: int = 8,
                  block_size: int = 16) -> Workload:
    """16 sequences, each with `ctx` cached tokens (a number, or one per
    sequence) and a `chunk`-token causal query chunk at positions
    ctx .. ctx+chunk-1 whose K/V are first written by the slot writer;
    64/8 heads, d=128, b=16 unless given, random placement."""
    rng = np.random.default_rng(seed + 1000)
    b = block_size
    ctx_lens = np.full(batch, ctx, dtype=np.int32) if np.isscalar(ctx) else np.asarray(ctx, np.int32)
    total = ctx_lens.astype(np.int64) + chunk
    counts = [_blocks_for(int(L), b) for L in total]
    tables = _tables_from_counts(counts, rng.permutation(num_blocks).astype(np.int32))
    seq_idx = np.repeat(np.arange(batch, dtype=np.int32), chunk)
    positions = (ctx_lens.astype(np.int64)[:, None] + np.arange(chunk, dtype=np.int64)[None, :]).ravel()
    return Workload("prefill_chunk", "prefill", num_q_heads, num_kv_heads, 128, b, num_blocks, 1.0 / math.sqrt(128),
                    total.astype(np.int32), tables, _referenced(tables), seed,
                    new_seq_idx=seq_idx, new_positions=positions, ctx_lens=ctx_lens, chunk=chunk)


def custom(lens, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
           num_blocks: Optional[int] = None, seed: int = SEED_BASE + 100, name: str = "custom",
           partition_tokens: int = 0) -> Workload:
    """Decode batch with the given sequence lengths (zeros allowed), random
    placement in a pool with spare blocks, scale 1/sqrt(head_dim)."""
    rng = np.random.default_rng(seed)
    b = block_size
    counts = [_blocks_for(int(L), b) for L in lens]
    nb = num_blocks if num_blocks is not None else max(8, 2 * sum(counts) + 3)
    tables = _tables_from_counts(counts, rng.permutation(nb).astype(np.int32))
    seq = np.asarray(lens, dtype=np.int32)
    has = seq > 0
    return Workload(name, "decode", num_q_heads, num_kv_heads, head_dim, b, nb, 1.0 / math.sqrt(head_dim),
                    seq, tables, _referenced(tables), seed,
                    new_seq_idx=np.nonzero(has)[0].astype(np.int32),
                    new_positions=seq[has].astype(np.int64) - 1, partition_tokens=partition_tokens)


def shared_groups(prefix_lens, suffix_lens, group_size: int, num_q_heads: int, num_kv_heads: int,
                  head_dim: int = 128, block_size: int = 16, seed: int = SEED_BASE + 200,
                  name: str = "shared_groups") -> Workload:
    """Decode batch of len(prefix_lens) groups of ``group_size`` consecutive
    sequences.  The tables of group i start with the same prefix_lens[i] // b
    physical blocks (prefix_lens are whole blocks); sequence k of the group
    then holds suffix_lens[i * group_size + k] tokens in private blocks.
    Random placement, a pool with spare blocks, scale 1/sqrt(head_dim)."""
    rng = np.random.default_rng(seed)
    b = block_size
    prefix_lens = [int(x) for x in prefix_lens]
    suffix_lens = [int(x) for x in suffix_lens]
    assert all(p % b == 0 for p in prefix_lens) and len(suffix_lens) == len(prefix_lens) * group_size
    B = len(suffix_lens)
    lens = np.asarray([prefix_lens[s // group_size] + suffix_lens[s] for s in range(B)], dtype=np.int32)
    need = sum(p // b for p in prefix_lens) + sum(_blocks_for(x, b) for x in suffix_lens)
    nb = max(8, 2 * need + 3)
    ids = iter(rng.permutation(nb).astype(np.int32).tolist())
    width = max(1, max(_blocks_for(int(L), b) for L in lens))
    tables = np.full((B, width), -1, dtype=np.int32)
    for gi, plen in enumerate(prefix_lens):
        shared = [next(ids) for _ in range(plen // b)]
        for k in range(group_size):
            s = gi * group_size + k
            own = [next(ids) for _ in range(_blocks_for(suffix_lens[s], b))]
            row = shared + own
            tables[s, :len(row)] = row
    has = lens > 0
    return Workload(name, "decode", num_q_heads, num_kv_heads, head_dim, b, nb, 1.0 / math.sqrt(head_dim),
                    lens, tables, _referenced(tables), seed,
                    new_seq_idx=np.nonzero(has)[0].astype(np.int32),
                    new_positions=lens[has].astype(np.int64) - 1,
                    notes={"prefix_lens": np.asarray(prefix_lens, np.int32), "group_size": group_size})


CONFIGS = {
    "tiny": tiny,
    "tiny_page_example": tiny_page_example,
    "llama70b_decode": llama70b_decode,
    "long_context": long_context,
    "shared_prefix": shared_prefix,
    "beam_fork": beam_fork,
    "prefill_chunk": prefill_chunk,
}


# ---------------------------------------------------------------------------
# tensors
# ---------------------------------------------------------------------------

def _generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_tensors(w: Workload, device="cpu", chunk_rows: int = 2048) -> Dict[str, torch.Tensor]:
    """Random bf16 tensors for a workload, created on ``device``.

    pool    [NB][2][Hkv][b][d]  referenced blocks ~ N(0,1), all others zero
    q       [B][Hq][d] (decode) or [B][C][Hq][d] (prefill)
    new_k, new_v [N][Hkv][d]    the tokens the slot writer stores
    """
    device = torch.device(device)
    g = _generator(device, w.seed)
    H, b, d = w.num_kv_heads, w.block_size, w.head_dim
    pool = torch.zeros((w.num_blocks, 2, H, b, d), dtype=torch.bfloat16, device=device)
    ids = torch.as_tensor(w.referenced, dtype=torch.int64, device=device)
    for start in range(0, ids.numel(), chunk_rows):
        sel = ids[start:start + chunk_rows]
        pool[sel] = randn_bf16((sel.numel(), 2, H, b, d), g, device)
    if w.kind == "prefill":
        q = randn_bf16((w.batch, w.chunk, w.num_q_heads, d), g, device)
    else:
        q = randn_bf16((w.batch, w.num_q_heads, d), g, device)
    n_new = 0 if w.new_positions is None else len(w.new_positions)
    new_k = randn_bf16((n_new, H, d), g, device)
    new_v = randn_bf16((n_new, H, d), g, device)
    return {"pool": pool, "q": q, "new_k": new_k, "new_v": new_v}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
