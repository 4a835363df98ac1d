"""Reference model of a block manager with a prefix cache -- TEST INFRASTRUCTURE.

Only ``tests/`` may import this module.  It shares nothing with the library's
block manager (``paged_kv_cache_167_gb300/csrc/pa_block_manager.cpp``): it
keys a cached block by the whole token prefix that ends with it, a plain
dictionary of tuples, where the library chains entries to their parents.

What it states (how-pagedattention-works (aiinfrainterviews.com), the
shared-system-prompt paragraph and feature table; auto-20261007-1900-en
(lihaoran.work), "Shared prefixes need matching computation"):

* a block's K/V are a function of every token up to its end and of the
  conditions of the computation, so block i of a request may reuse a cached
  block only when the condition and tokens[0 : (i+1)*b] are equal -- the same
  tokens after another context do not match;
* a prefix shared by many requests is held once; every table points at it and
  each block counts its holders (the cache holds one reference);
* only whole blocks are cached; matching stops at the first block not cached.

Readings where the pages are silent (the library's header states the same):
eviction takes, among entries whose block nothing but the cache holds, the one
used least recently, and removes with it every entry whose prefix extends its
prefix; a use stamps the blocks of one chain deepest first, so a prefix is
never older than its extensions; an allocation that finds no free block
evicts first; publishing keeps an existing entry for equal content and stops
at a block the cache already holds under other content.

Block identities here are opaque integers that are never reused; tests compare
the library's tables with the model's through the sharing structure.
"""
from __future__ import annotations

from typing import Dict, List, Tuple


class NoBlocks(Exception):
    pass


class PrefixCacheModel:
    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks, self.b = num_blocks, block_size
        self.ref: Dict[int, int] = {}                       # block -> holders (sequences and the cache)
        self.entries: Dict[tuple, List[int]] = {}           # (condition, prefix tokens) -> [block, tick]
        self.key_of_block: Dict[int, tuple] = {}
        self.seqs: Dict[int, Tuple[List[int], int]] = {}    # seq -> (blocks, tokens)
        self.clock = 0
        self._next_block = 0
        self._next_seq = 0
        self.hit_tokens = self.query_tokens = 0

    # -- counts ----------------------------------------------------------------
    def num_free(self) -> int:
        return self.num_blocks - len(self.ref)

    def evictable(self) -> List[tuple]:
        return [k for k, (blk, _) in self.entries.items() if self.ref[blk] == 1]

    def available(self) -> int:
        return self.num_free() + len(self.evictable())

    # -- blocks ------------------------------------------------------------------
    def _release(self, blk: int) -> None:
        self.ref[blk] -= 1
        if self.ref[blk] == 0:
            del self.ref[blk]

    def _evict_oldest(self) -> int:
        cands = self.evictable()
        if not cands:
            return 0
        victim = min(cands, key=lambda k: self.entries[k][1])
        cond, prefix = victim
        before = self.num_free()
        for k in [k for k in self.entries if k[0] == cond and k[1][:len(prefix)] == prefix]:
            blk = self.entries.pop(k)[0]
            del self.key_of_block[blk]
            self._release(blk)
        return self.num_free() - before

    def _alloc(self) -> int:
        if self.num_free() == 0:
            self._evict_oldest()
        blk = self._next_block
        self._next_block += 1
        self.ref[blk] = 1
        return blk

    def _stamp(self, chain: List[tuple]) -> None:
        for k in reversed(chain):
            self.clock += 1
            self.entries[k][1] = self.clock

    # -- sequences ---------------------------------------------------------------
    def _new_seq(self, blocks: List[int], tokens: int) -> int:
        sid = self._next_seq
        self._next_seq += 1
        self.seqs[sid] = (blocks, tokens)
        return sid

    def add_seq(self) -> int:
        return self._new_seq([], 0)

    def match_chain(self, tokens, condition: int) -> List[tuple]:
        chain = []
        for i in range(len(tokens) // self.b):
            key = (condition, tuple(tokens[:(i + 1) * self.b]))
            if key not in self.entries:
                break
            chain.append(key)
        return chain

    def prefix_match(self, tokens, condition: int = 0) -> int:
        return len(self.match_chain(tokens, condition)) * self.b

    def add_seq_cached(self, tokens, condition: int = 0) -> Tuple[int, int]:
        chain = self.match_chain(tokens, condition)
        blocks = [self.entries[k][0] for k in chain]
        for blk in blocks:
            self.ref[blk] += 1
        self._stamp(chain)
        matched = len(chain) * self.b
        self.hit_tokens += matched
        self.query_tokens += len(tokens)
        return self._new_seq(blocks, matched), matched

    def cache_seq(self, sid: int, tokens, condition: int = 0) -> int:
        blocks, n = self.seqs[sid]
        if len(tokens) > n:
            raise ValueError("more tokens than the sequence holds")
        chain, inserted = [], 0
        for i in range(len(tokens) // self.b):
            key = (condition, tuple(tokens[:(i + 1) * self.b]))
            if key not in self.entries:
                blk = blocks[i]
                if blk in self.key_of_block:
                    break
                self.entries[key] = [blk, 0]
                self.key_of_block[blk] = key
                self.ref[blk] += 1
                inserted += 1
            chain.append(key)
        self._stamp(chain)
        return inserted

    def append(self, sid: int, n: int):
        """Returns the copy-on-write pair (src, dst) or None; raises NoBlocks."""
        blocks, tokens = self.seqs[sid]
        b = self.b
        fresh = -(-(tokens + n) // b) - len(blocks)
        cow = n > 0 and tokens % b != 0 and self.ref[blocks[-1]] > 1
        if self.available() < fresh + int(cow):
            raise NoBlocks()
        pair = None
        if cow:
            src = blocks[-1]
            dst = self._alloc()
            self._release(src)
            blocks[-1] = dst
            pair = (src, dst)
        for _ in range(fresh):
            blocks.append(self._alloc())
        self.seqs[sid] = (blocks, tokens + n)
        return pair

    def fork(self, sid: int) -> int:
        blocks, tokens = self.seqs[sid]
        for blk in blocks:
            self.ref[blk] += 1
        return self._new_seq(list(blocks), tokens)

    def free_seq(self, sid: int) -> None:
        blocks, _ = self.seqs.pop(sid)
        for blk in blocks:
            self._release(blk)

    def evict(self, n_blocks: int) -> int:
        freed = 0
        while freed < n_blocks and self.evictable():
            freed += self._evict_oldest()
        return freed
