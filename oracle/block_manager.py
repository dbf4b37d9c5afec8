"""Block manager model: free-block FIFO, ref_cnt, block tables — test infrastructure only.

Sources:

* "PagedAttention: manage the KV cache like virtual memory", §3.2: the pool keeps a
  free-block queue; allocation pops from its head and freeing pushes to its tail;
  every block carries a reference count.  §3.3: admission pops enough free blocks for
  the prompt; each decode token fills the current last block and a full block makes
  the sequence pop one more; finishing decrements every block's count and a block is
  really freed when its count reaches 0.  §2/§3.5: a block is free (count 0) or owned
  (count > 0).  §4: admission succeeds while enough free blocks remain.
* "Lecture 33 — KV Cache management", §2.2 (per-sequence block table, slot address)
  and §2.4 (fork copies only the table and raises each block's count; a write into a
  block whose count is above 1 first takes a new block, copies the old block into
  it, points the writer's table at it and lowers the old block's count).  §5.2
  (preemption by swapping): the victim's blocks are copied to host memory, its device
  blocks are released for the others, and when memory frees up the blocks are copied
  back and the sequence resumes.

Readings where the pages are silent:

* A sequence's blocks are released in table order when it is freed.
* ``import_seq`` claims named blocks directly (used to set up synthetic states such
  as two sequences sharing a block); a claimed free block leaves the free queue.
* Running out of free blocks raises ``NoBlocks`` and leaves the state unchanged.
* Swapping: the host swap space is a second pool of blocks with its own FIFO queue.
  Swap-out gives each table entry, in order, a host block, then releases the device
  blocks in table order exactly as ``free`` does (a block shared with another
  sequence stays for it; the swapped sequence takes its own host copy).  Swap-in pops
  one device block per table entry in order and returns the host blocks to the host
  queue's tail in table order.  A swapped sequence can only be freed or swapped in.

Prefix caching ("PagedAttention: manage the KV cache like virtual memory" §3.4–§3.5;
"Lecture 33" §6.2–§6.3): a full block is named by its parent's name and its tokens, so a
name stands for the whole token prefix up to the block's end.  The model keys blocks by that
exact prefix (a tuple of token ids), so it never confuses two prefixes; ``block_hash``
computes the 64-bit FNV-1a chain the library publishes for the same key.  Admission matches
the prompt's full blocks in order and stops at the first miss; a hit raises the block's count
and takes it out of the free queue if nobody held it; the other blocks are popped and the new
full ones registered.  A popped block loses its registration (new contents).  Readings: the
first block's parent name is the FNV offset basis; blocks filled during decode are not
registered (token ids are not known there).
"""
from __future__ import annotations

from collections import deque
from typing import Dict, List, Optional, Sequence, Tuple

FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3


def fnv1a64(data: bytes, h: int = FNV64_OFFSET) -> int:
    """64-bit FNV-1a: for each byte, xor it in, then multiply by the FNV prime (mod 2^64)."""
    for byte in data:
        h ^= byte
        h = (h * FNV64_PRIME) & 0xFFFFFFFFFFFFFFFF
    return h


def block_hash(parent: int, tokens: Sequence[int]) -> int:
    """Name of a full block: FNV-1a over the parent's name (8 bytes little-endian) then the
    token ids (4 bytes little-endian each)."""
    data = parent.to_bytes(8, "little") + b"".join((int(t) & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


def prefix_hash(prefix: Sequence[int], block_size: int) -> int:
    """Name of the last full block of ``prefix`` (len a multiple of block_size)."""
    h = FNV64_OFFSET
    for i in range(0, len(prefix), block_size):
        h = block_hash(h, prefix[i:i + block_size])
    return h


class BlockManagerError(Exception):
    pass


class NoBlocks(BlockManagerError):
    pass


class InvalidArg(BlockManagerError):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free_queue = deque(range(num_blocks))   # head = next to allocate
        self.ref_cnt = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.num_tokens: Dict[int, int] = {}
        self.host_free: deque = deque()
        self.swapped: Dict[int, bool] = {}
        self.cached: Dict[tuple, int] = {}         # token prefix -> block holding its last full block
        self.block_key: Dict[int, tuple] = {}      # registered block -> its prefix

    # -- pool ---------------------------------------------------------------------------
    def num_free(self) -> int:
        return len(self.free_queue)

    def _pop(self) -> int:
        if not self.free_queue:
            raise NoBlocks("free block queue is empty")
        b = self.free_queue.popleft()
        assert self.ref_cnt[b] == 0
        self.ref_cnt[b] = 1
        key = self.block_key.pop(b, None)          # new contents: the cached prefix is gone
        if key is not None and self.cached.get(key) == b:
            del self.cached[key]
        return b

    def _release(self, b: int) -> None:
        assert self.ref_cnt[b] > 0
        self.ref_cnt[b] -= 1
        if self.ref_cnt[b] == 0:
            self.free_queue.append(b)

    # -- sequences ----------------------------------------------------------------------
    def import_seq(self, seq: int, blocks: Sequence[int], n_tokens: int) -> None:
        if seq in self.tables:
            raise InvalidArg("sequence exists")
        if len(blocks) != -(-n_tokens // self.block_size):
            raise InvalidArg("block count does not cover n_tokens")
        for b in blocks:
            if not 0 <= b < self.num_blocks:
                raise InvalidArg("block id out of range")
        for b in blocks:
            if self.ref_cnt[b] == 0:
                self.free_queue.remove(b)
            self.ref_cnt[b] += 1
        self.tables[seq] = list(blocks)
        self.num_tokens[seq] = n_tokens

    def allocate(self, seq: int, n_tokens: int) -> None:
        """Admit a sequence with an ``n_tokens`` prompt: pop ceil(n / B) blocks."""
        if seq in self.tables:
            raise InvalidArg("sequence exists")
        need = -(-n_tokens // self.block_size)
        if need > len(self.free_queue):
            raise NoBlocks("not enough free blocks")
        self.tables[seq] = [self._pop() for _ in range(need)]
        self.num_tokens[seq] = n_tokens

    def _resident(self, seq: int) -> List[int]:
        if seq not in self.tables or self.swapped.get(seq):
            raise InvalidArg("not a resident sequence")
        return self.tables[seq]

    def allocate_cached(self, seq: int, tokens: Sequence[int]) -> int:
        """Admit a prompt, re-using the blocks of its longest cached full-block prefix;
        returns the number of cached tokens."""
        if seq in self.tables:
            raise InvalidArg("sequence exists")
        bs = self.block_size
        tokens = [int(t) for t in tokens]
        n_full, need = len(tokens) // bs, -(-len(tokens) // bs)
        keys = [tuple(tokens[:(i + 1) * bs]) for i in range(n_full)]
        hits = []
        for k in keys:
            b = self.cached.get(k)
            if b is None:
                break
            hits.append(b)
        held_free = sum(1 for b in hits if self.ref_cnt[b] == 0)
        if need - len(hits) > len(self.free_queue) - held_free:
            raise NoBlocks("not enough free blocks")
        table = []
        for b in hits:
            if self.ref_cnt[b] == 0:
                self.free_queue.remove(b)
            self.ref_cnt[b] += 1
            table.append(b)
        for i in range(len(hits), need):
            b = self._pop()
            table.append(b)
            if i < n_full and keys[i] not in self.cached:
                self.cached[keys[i]] = b
                self.block_key[b] = keys[i]
        self.tables[seq] = table
        self.num_tokens[seq] = len(tokens)
        return len(hits) * bs

    def block_hash(self, block: int) -> Optional[int]:
        key = self.block_key.get(block)
        return None if key is None else prefix_hash(key, self.block_size)

    def append_slot(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot of the sequence's next token; returns (slot, cow_pair or None)."""
        table = self._resident(seq)
        p = self.num_tokens[seq]
        bs = self.block_size
        cow = None
        if p % bs == 0:                      # last block full (or none yet): grow by one block
            table.append(self._pop())
        else:
            last = table[p // bs]
            if self.ref_cnt[last] > 1:       # shared: copy-on-write before the write
                new = self._pop()
                self.ref_cnt[last] -= 1
                table[p // bs] = new
                cow = (last, new)
        self.num_tokens[seq] = p + 1
        return table[p // bs] * bs + p % bs, cow

    def append_slots(self, seq: int, n: int) -> Tuple[List[int], List[Tuple[int, int]]]:
        """``n`` consecutive append_slot calls; all of them or none (state restored on NoBlocks)."""
        self._resident(seq)
        saved = (deque(self.free_queue), list(self.ref_cnt), {k: list(v) for k, v in self.tables.items()},
                 dict(self.num_tokens))
        slots, cows = [], []
        try:
            for _ in range(n):
                s, c = self.append_slot(seq)
                slots.append(s)
                if c is not None:
                    cows.append(c)
        except NoBlocks:
            self.free_queue, self.ref_cnt, self.tables, self.num_tokens = saved
            raise
        return slots, cows

    def fork(self, parent: int, child: int) -> None:
        if child in self.tables:
            raise InvalidArg("sequence exists")
        self.tables[child] = list(self._resident(parent))
        self.num_tokens[child] = self.num_tokens[parent]
        for b in self.tables[child]:
            self.ref_cnt[b] += 1

    def free(self, seq: int) -> None:
        if self.swapped.pop(seq, False):
            self.host_free.extend(self.tables.pop(seq))
        else:
            for b in self.tables.pop(seq):
                self._release(b)
        del self.num_tokens[seq]

    # -- swapping ------------------------------------------------------------------------
    def set_host_pool(self, num_host_blocks: int) -> None:
        if any(self.swapped.values()):
            raise InvalidArg("a sequence is swapped out")
        self.host_free = deque(range(num_host_blocks))

    def swap_out(self, seq: int) -> List[Tuple[int, int]]:
        if self.swapped.get(seq) or seq not in self.tables:
            raise InvalidArg("not a resident sequence")
        table = self.tables[seq]
        if len(table) > len(self.host_free):
            raise NoBlocks("host swap space is full")
        host = [self.host_free.popleft() for _ in table]
        pairs = list(zip(table, host))
        for b in table:
            self._release(b)
        self.tables[seq] = host
        self.swapped[seq] = True
        return pairs

    def swap_in(self, seq: int) -> List[Tuple[int, int]]:
        if not self.swapped.get(seq):
            raise InvalidArg("not swapped out")
        host = self.tables[seq]
        if len(host) > len(self.free_queue):
            raise NoBlocks("not enough free device blocks")
        dev = [self._pop() for _ in host]
        self.host_free.extend(host)
        self.tables[seq] = dev
        self.swapped[seq] = False
        return list(zip(host, dev))

    def export(self, seqs: Sequence[int], max_blocks: int) -> Tuple[List[List[int]], List[int]]:
        """Block tables padded with -1 to ``max_blocks`` and the token counts."""
        tables, lens = [], []
        for s in seqs:
            t = self._resident(s)
            if len(t) > max_blocks:
                raise InvalidArg("table longer than max_blocks")
            tables.append(t + [-1] * (max_blocks - len(t)))
            lens.append(self.num_tokens[s])
        return tables, lens
