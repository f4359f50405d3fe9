"""Plain-Python model of the host KV block manager's policy.

TEST INFRASTRUCTURE ONLY (see the package docstring).  It is an independent
second implementation of the same policy as the C++ manager in the product
library; the tests require both to produce identical block tables, slot
mappings, copy-on-write pairs and reference counts.

Policy, from the pages:
  - wywy.jp notes, "KV cache manager" and the parallel-sampling walkthrough:
    one preallocated pool split into physical blocks; per-sequence block tables
    map logical to physical blocks; each physical block carries a reference
    count; when a sequence must write into its last logical block and that
    block's count is above one, a new block is allocated, the block engine
    copies the old contents into it and the count drops by one; the last
    remaining holder writes in place.
  - zhaifeiyue.github.io detail page, "Memory Management" table: Allocate when
    the previous logical block is full (one physical block), Free the whole
    request's blocks when it finishes or is preempted, Copy-on-Write one block
    when writing a block whose count exceeds one.
  - ricepunchb garden, section 3.2: slot = table[pos // B] * B + pos % B.

Readings where the pages are silent (both implementations follow them):
  - the free list starts as a seeded permutation of all block ids, made by a
    Fisher-Yates shuffle driven by SplitMix64 (Steele, Lea and Flood, OOPSLA
    2014), draws j = next() mod (i + 1) for i = n-1 .. 1;
  - allocation pops the front of the free list; freeing pushes a block whose
    count reached zero to the back, in block-table order;
  - fork increments the count of every block of the parent's table, the
    partial last block included;
  - a failing operation leaves the state unchanged (out of blocks -> OOM).
"""
from __future__ import annotations

from collections import deque

MASK64 = (1 << 64) - 1


class OutOfBlocks(Exception):
    pass


class InvalidRequest(Exception):
    pass


def splitmix64_stream(seed: int):
    """SplitMix64: add the golden-gamma constant, then two xor-shift-multiply rounds."""
    state = seed & MASK64
    while True:
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def seeded_permutation(n: int, seed: int) -> list:
    """Fisher-Yates over [0, n) drawing from SplitMix64(seed)."""
    a = list(range(n))
    rng = splitmix64_stream(seed)
    for i in range(n - 1, 0, -1):
        j = next(rng) % (i + 1)
        a[i], a[j] = a[j], a[i]
    return a


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int, seed: int):
        if num_blocks <= 0 or block_size <= 0:
            raise InvalidRequest("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.B = block_size
        self.free = deque(seeded_permutation(num_blocks, seed))
        self.ref = [0] * num_blocks
        self.tables = {}   # seq_id -> list of physical block ids (CPU ids while swapped)
        self.ctx = {}      # seq_id -> number of tokens written
        self.swapped = {}  # seq_id -> True while the sequence's blocks are in the CPU pool
        self.num_cpu_blocks = 0
        self.cpu_free = deque()
        self.cpu_ref = []

    # -- queries ---------------------------------------------------------
    def num_free(self) -> int:
        return len(self.free)

    def refcount(self, block: int) -> int:
        return self.ref[block]

    def block_table(self, seq_id: int) -> list:
        if seq_id not in self.tables:
            raise InvalidRequest("unknown sequence")
        return list(self.tables[seq_id])

    def context_len(self, seq_id: int) -> int:
        if seq_id not in self.ctx:
            raise InvalidRequest("unknown sequence")
        return self.ctx[seq_id]

    # -- operations ------------------------------------------------------
    def _slot(self, table: list, pos: int) -> int:
        return table[pos // self.B] * self.B + pos % self.B

    def _take(self) -> int:
        blk = self.free.popleft()
        self.ref[blk] = 1
        return blk

    def add_sequence(self, seq_id: int, prompt_len: int) -> list:
        """Allocate ceil(prompt_len / B) blocks; return the prompt tokens' slots."""
        if seq_id in self.tables or prompt_len < 0:
            raise InvalidRequest("sequence exists or negative length")
        need = -(-prompt_len // self.B)
        if need > len(self.free):
            raise OutOfBlocks()
        table = [self._take() for _ in range(need)]
        self.tables[seq_id] = table
        self.ctx[seq_id] = prompt_len
        self.swapped[seq_id] = False
        return [self._slot(table, p) for p in range(prompt_len)]

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.tables or child in self.tables or self.swapped[parent]:
            raise InvalidRequest("unknown or swapped-out parent, or existing child")
        table = list(self.tables[parent])
        for blk in table:
            self.ref[blk] += 1
        self.tables[child] = table
        self.ctx[child] = self.ctx[parent]
        self.swapped[child] = False

    def append_slot(self, seq_id: int):
        """Reserve the slot of the sequence's next token.

        Returns (slot, cow_src, cow_dst); cow_src = cow_dst = -1 when no copy
        is needed.
        """
        if seq_id not in self.tables or self.swapped[seq_id]:
            raise InvalidRequest("unknown or swapped-out sequence")
        table = self.tables[seq_id]
        pos = self.ctx[seq_id]
        src = dst = -1
        if pos % self.B == 0:
            # previous logical block full (or none yet): allocate a fresh block
            if not self.free:
                raise OutOfBlocks()
            table.append(self._take())
        else:
            last = table[-1]
            if self.ref[last] > 1:
                # shared partially filled block: copy-on-write
                if not self.free:
                    raise OutOfBlocks()
                new = self._take()
                self.ref[last] -= 1
                table[-1] = new
                src, dst = last, new
        self.ctx[seq_id] = pos + 1
        return self._slot(table, pos), src, dst

    def free_sequence(self, seq_id: int) -> None:
        if seq_id not in self.tables:
            raise InvalidRequest("unknown sequence")
        ref, free = (self.cpu_ref, self.cpu_free) if self.swapped[seq_id] else (self.ref, self.free)
        for blk in self.tables.pop(seq_id):
            ref[blk] -= 1
            if ref[blk] == 0:
                free.append(blk)
        del self.ctx[seq_id]
        del self.swapped[seq_id]

    # -- swapping (wywy.jp notes: "Swapping", all-or-nothing eviction) ---------
    def add_cpu_pool(self, num_cpu_blocks: int, seed: int) -> None:
        if self.num_cpu_blocks or num_cpu_blocks <= 0:
            raise InvalidRequest("CPU pool exists or has no blocks")
        self.num_cpu_blocks = num_cpu_blocks
        self.cpu_free = deque(seeded_permutation(num_cpu_blocks, seed))
        self.cpu_ref = [0] * num_cpu_blocks

    def _swap(self, seq_ids, out: bool):
        if not self.num_cpu_blocks:
            raise InvalidRequest("no CPU pool")
        if len(set(seq_ids)) != len(seq_ids):
            raise InvalidRequest("repeated sequence")
        for sid in seq_ids:
            if sid not in self.tables or self.swapped[sid] == out:
                raise InvalidRequest("unknown sequence or already in the target pool")
        uses = {}
        for sid in seq_ids:
            for blk in self.tables[sid]:
                uses[blk] = uses.get(blk, 0) + 1     # dict keeps first-seen order
        src_ref, src_free = (self.ref, self.free) if out else (self.cpu_ref, self.cpu_free)
        dst_ref, dst_free = (self.cpu_ref, self.cpu_free) if out else (self.ref, self.free)
        if any(src_ref[b] != n for b, n in uses.items()):
            raise InvalidRequest("a block is shared outside the group")
        if len(uses) > len(dst_free):
            raise OutOfBlocks()
        moved, pairs = {}, []
        for blk in uses:
            new = dst_free.popleft()
            dst_ref[new] = src_ref[blk]
            moved[blk] = new
            pairs.append((blk, new))
        for blk in uses:
            src_ref[blk] = 0
            src_free.append(blk)
        for sid in seq_ids:
            self.tables[sid] = [moved[b] for b in self.tables[sid]]
            self.swapped[sid] = out
        return pairs

    def swap_out(self, seq_ids) -> list:
        """Move a group of resident sequences to the CPU pool; returns (gpu, cpu) pairs."""
        return self._swap(list(seq_ids), True)

    def swap_in(self, seq_ids) -> list:
        """Move a group of swapped-out sequences back; returns (cpu, gpu) pairs."""
        return self._swap(list(seq_ids), False)
