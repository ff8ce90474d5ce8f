"""Plain-Python model of the host-side KV-cache page manager.

TEST INFRASTRUCTURE ONLY: imported by the tests and by the benchmark's
CPU-baseline leg; the product library never imports or calls it, and it
shares no code with the native manager.

What it follows (page "TensorRT-LLM框架解析与高性能推理优化实践"):
  * §4.1 / §4.2 "KV缓存管理细节": K/V live in fixed-size blocks of one pool;
    a manager hands blocks to sequences (allocate / free) and keeps, per
    sequence, the list of its blocks, which is the block table the attention
    kernel walks.  Blocks may be reused and prefixes shared (§4.1, the
    manager's duties).
  * §5.2 "抢占策略实现": when the pool cannot hold a request, running
    requests are preempted last-in-first-out: the most recently admitted one
    gives back its blocks first, until the request fits or nothing is left.
Where the page leaves a choice open, this model fixes it (the native manager
follows the same rules, so the two agree id for id):
  * free blocks form a stack; the pool starts with block 0 on top, an
    allocation pops the top, a release pushes the block;
  * a sequence forked from another shares the parent's first ceil(n / P)
    blocks (reference counts); a shared block is copied before a sequence
    writes into it (copy-on-write): a fresh block is popped, the pair
    (old, new) is reported for the caller to copy on the device, and the
    writer's table points at the new block;
  * an append of several sequences is all-or-nothing: if the pool cannot
    supply every block it needs (new pages and copies), nothing changes;
  * releasing a sequence pushes its blocks last page first, and a block
    returns to the free stack when its count reaches zero;
  * preemption frees whole sequences in reverse admission order, skipping
    the protected ones; if even that cannot free enough, nothing changes.
"""
from __future__ import annotations

import numpy as np

OK = 0
ERR_INVALID_ARG = 1
ERR_OUT_OF_BLOCKS = 7


class KVCacheManagerModel:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        if num_blocks <= 0 or block_size <= 0 or max_blocks_per_seq <= 0:
            raise ValueError("sizes must be positive")
        self.N, self.P, self.M = num_blocks, block_size, max_blocks_per_seq
        self.free = list(range(num_blocks - 1, -1, -1))   # top of stack = end
        self.ref = [0] * num_blocks
        self.seqs = {}          # seq_id -> [pages list, length, admission number]
        self.admitted = 0

    # -- queries ----------------------------------------------------------
    def num_free(self) -> int:
        return len(self.free)

    def length(self, seq_id: int) -> int:
        return self.seqs[seq_id][1]

    def pages(self, seq_id: int):
        return list(self.seqs[seq_id][0])

    def block_tables(self, seq_ids):
        """int32 [n, M] tables (-1 past the last page) and int32 [n] lengths."""
        n = len(seq_ids)
        tab = np.full((n, self.M), -1, np.int32)
        lens = np.zeros(n, np.int32)
        for r, s in enumerate(seq_ids):
            pg, L, _ = self.seqs[s]
            tab[r, :len(pg)] = pg
            lens[r] = L
        return tab, lens

    # -- sequence life cycle ----------------------------------------------
    def add(self, seq_id: int) -> int:
        if seq_id in self.seqs or seq_id < 0:
            return ERR_INVALID_ARG
        self.seqs[seq_id] = [[], 0, self.admitted]
        self.admitted += 1
        return OK

    def fork(self, parent: int, child: int, num_tokens: int) -> int:
        """child starts as the first num_tokens tokens of parent, sharing pages."""
        if parent not in self.seqs or child in self.seqs or child < 0:
            return ERR_INVALID_ARG
        ppages, plen, _ = self.seqs[parent]
        if num_tokens < 0 or num_tokens > plen:
            return ERR_INVALID_ARG
        shared = ppages[:-(-num_tokens // self.P)] if num_tokens else []
        for b in shared:
            self.ref[b] += 1
        self.seqs[child] = [list(shared), num_tokens, self.admitted]
        self.admitted += 1
        return OK

    def release(self, seq_id: int) -> int:
        if seq_id not in self.seqs:
            return ERR_INVALID_ARG
        pages = self.seqs.pop(seq_id)[0]
        for b in reversed(pages):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        return OK

    # -- append -------------------------------------------------------------
    def _plan(self, seq_ids, counts):
        """Blocks the append needs (new pages + copies), or None if invalid."""
        if len(set(seq_ids)) != len(seq_ids):
            return None
        ref_delta = {}
        need = 0
        for s, c in zip(seq_ids, counts):
            if s not in self.seqs or c < 0:
                return None
            pages, L, _ = self.seqs[s]
            if -(-(L + c) // self.P) > self.M:
                return None
            if c == 0:
                continue
            first = L // self.P                       # page of the first new token
            last = (L + c - 1) // self.P
            for j in range(first, last + 1):
                if j < len(pages):
                    b = pages[j]
                    if self.ref[b] + ref_delta.get(b, 0) > 1:   # shared: copy first
                        ref_delta[b] = ref_delta.get(b, 0) - 1
                        need += 1
                else:
                    need += 1
        return need

    def blocks_needed(self, seq_ids, counts):
        need = self._plan(seq_ids, counts)
        return -1 if need is None else need

    def append(self, seq_ids, counts):
        """Reserve slots for counts[i] new tokens of seq_ids[i], in order.

        Returns (status, slot_mapping int64 [sum counts], copies int32 [k, 2])."""
        empty = (np.zeros(0, np.int64), np.zeros((0, 2), np.int32))
        need = self._plan(seq_ids, counts)
        if need is None:
            return (ERR_INVALID_ARG,) + empty
        if need > len(self.free):
            return (ERR_OUT_OF_BLOCKS,) + empty
        slots, copies = [], []
        for s, c in zip(seq_ids, counts):
            rec = self.seqs[s]
            pages = rec[0]
            for _ in range(c):
                pos = rec[1]
                j = pos // self.P
                if j == len(pages):
                    b = self.free.pop()
                    self.ref[b] = 1
                    pages.append(b)
                elif self.ref[pages[j]] > 1:
                    old = pages[j]
                    b = self.free.pop()
                    self.ref[b] = 1
                    self.ref[old] -= 1
                    pages[j] = b
                    copies.append((old, b))
                slots.append(pages[j] * self.P + pos % self.P)
                rec[1] = pos + 1
        return (OK, np.array(slots, np.int64),
                np.array(copies, np.int32).reshape(-1, 2))

    # -- preemption -----------------------------------------------------------
    def preempt_for(self, needed: int, protected=()):
        """Free whole sequences, most recently admitted first, until at least
        `needed` blocks are free.  Returns (status, victims in order)."""
        if needed < 0:
            return ERR_INVALID_ARG, []
        prot = set(protected)
        order = sorted((rec[2], s) for s, rec in self.seqs.items() if s not in prot)
        ref_delta = {}
        free = len(self.free)
        victims = []
        for _, s in reversed(order):
            if free >= needed:
                break
            for b in self.seqs[s][0]:
                ref_delta[b] = ref_delta.get(b, 0) - 1
                if self.ref[b] + ref_delta[b] == 0:
                    free += 1
            victims.append(s)
        if free < needed:
            return ERR_OUT_OF_BLOCKS, []
        for s in victims:
            self.release(s)
        return OK, victims
