"""Prefix caching of the host block manager against its oracle model (CPU).

Sources: "PagedAttention: manage the KV cache like virtual memory" §3.4–§3.5 (a full block is
named by a hash of its parent's hash and its tokens; a hit touches the block, which may sit in
the free queue as an eviction candidate; three block states) and "Lecture 33 — KV Cache
management" §6.1–§6.3 (a long shared system prompt; cached free blocks are taken out of the
middle of a doubly linked free queue in O(1)).
"""
import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, NoBlocks, fnv1a64, prefix_hash


def test_fnv1a64_matches_its_published_test_vectors():
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


class _Model:
    """The oracle's BlockManagerModel behind the product BlockManager's method names, so the
    closed-form cases below pin both without routing one through the other."""

    def __init__(self, num_blocks, block_size):
        self.m = BlockManagerModel(num_blocks, block_size)

    def __getattr__(self, name):
        return getattr(self.m, name)

    def ref_cnt(self, b):
        return self.m.ref_cnt[b]

    def free_queue(self):
        return list(self.m.free_queue)

    def num_cached(self):
        return len(self.m.cached)


def _product(num_blocks, block_size):
    from paged_kv_cache_160_gb300 import BlockManager
    return BlockManager(num_blocks, block_size)


MANAGERS = {"oracle": _Model, "product": _product}


@pytest.mark.parametrize("side", sorted(MANAGERS))
def test_system_prompt_is_computed_once(side):
    """Lecture 33 §6.1: a 3,000-token system prompt, then 10-token user turns.  Closed forms:
    188 = floor(3010 / 16) full blocks registered, 187 = floor(3000 / 16) of them shared,
    2,992 = 187 * 16 tokens reused."""
    rng = np.random.default_rng(0)
    system = [int(x) for x in rng.integers(0, 32000, 3000)]
    q1 = system + [int(x) for x in rng.integers(0, 32000, 10)]
    q2 = system + [int(x) for x in rng.integers(0, 32000, 10)]
    bs = 16
    bm = MANAGERS[side](400, bs)
    assert bm.allocate_cached(1, q1) == 0                    # cold: everything is computed
    assert bm.num_cached() == 188                            # its 188 full blocks are registered
    assert bm.allocate_cached(2, q2) == 2992                 # 187 shared blocks: 2,992 tokens reused
    (t1, t2), lens = bm.export([1, 2], 200)
    assert lens == [3010, 3010]
    assert t1[:187] == t2[:187] and t1[187] != t2[187]
    assert all(bm.ref_cnt(b) == 2 for b in t1[:187]) and bm.ref_cnt(t1[187]) == 1
    # the hash of the last shared block names the whole 2,992-token prefix
    assert bm.block_hash(t1[186]) == prefix_hash(system[:2992], bs)
    bm.free(1)
    bm.free(2)                                               # cached and free: ref 0, hash kept
    assert all(bm.ref_cnt(b) == 0 and bm.block_hash(b) is not None for b in t1[:187])
    queue = bm.free_queue()
    assert bm.allocate_cached(3, q1) == 3008                 # every full block of q1 is still cached
    # the hit blocks left the queue from its middle; only one new block was popped from the head
    rest = [b for b in queue if b not in set(t1[:188])]
    assert bm.free_queue() == rest[1:]


@pytest.mark.parametrize("side", sorted(MANAGERS))
def test_popping_a_cached_block_evicts_its_name(side):
    bm = MANAGERS[side](4, 2)
    assert bm.allocate_cached(0, [1, 2, 3, 4]) == 0          # blocks 0, 1 registered
    bm.free(0)                                               # queue: 2, 3, 0, 1
    assert bm.free_queue() == [2, 3, 0, 1]
    bm.allocate(1, 6)                                        # pops 2, 3, 0: block 0 gets new contents
    assert bm.block_hash(0) is None and bm.block_hash(1) is not None and bm.num_cached() == 1
    bm.free(1)                                               # queue: 1, 2, 3, 0
    assert bm.free_queue() == [1, 2, 3, 0]
    assert bm.allocate_cached(2, [1, 2, 3, 4]) == 0          # the chain breaks at its first block ...
    assert bm.export([2], 2)[0] == [[1, 2]] and bm.num_cached() == 2   # ... and is registered anew


@pytest.mark.parametrize("side", sorted(MANAGERS))
def test_a_prompt_shorter_than_a_block_is_never_cached(side):
    """Only full blocks are named: 15 tokens in 16-token blocks register nothing, and a second
    identical prompt reuses nothing."""
    bm = MANAGERS[side](8, 16)
    assert bm.allocate_cached(0, list(range(15))) == 0 and bm.num_cached() == 0
    assert bm.allocate_cached(1, list(range(15))) == 0
    assert bm.export([0, 1], 1)[0][0] != bm.export([0, 1], 1)[0][1]


def _ops(seed, n=2500):
    rng = np.random.default_rng(seed)
    prompts = [[int(x) for x in rng.integers(0, 50, int(rng.integers(1, 120)))] for _ in range(6)]
    ops, live, nxt = [], [], 0
    for _ in range(n):
        r = rng.random()
        if r < 0.3 or not live:
            base = prompts[int(rng.integers(0, len(prompts)))]
            cut = int(rng.integers(0, len(base) + 1))
            tail = [int(x) for x in rng.integers(0, 50, int(rng.integers(0, 40)))]
            ops.append(("allocate_cached", nxt, base[:cut] + tail)); live.append(nxt); nxt += 1
        elif r < 0.55:
            ops.append(("append_slot", int(rng.choice(live))))
        elif r < 0.62:
            ops.append(("fork", int(rng.choice(live)), nxt)); live.append(nxt); nxt += 1
        elif r < 0.68:
            ops.append(("swap_out", int(rng.choice(live))))
        elif r < 0.74:
            ops.append(("swap_in", int(rng.choice(live))))
        else:
            s = int(rng.choice(live)); ops.append(("free", s)); live.remove(s)
    return ops


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_prefix_cache_matches_oracle_model(seed):
    from paged_kv_cache_160_gb300 import BlockManager, NoBlocksError, PkvError
    nb, bs, nh = 120, 8, 60
    model, prod = BlockManagerModel(nb, bs), BlockManager(nb, bs)
    model.set_host_pool(nh)
    prod.set_host_pool(nh)
    live = set()
    hits = 0
    for op in _ops(seed):
        kind = op[0]
        if kind != "allocate_cached" and op[1] not in live:
            continue
        if kind in ("append_slot", "fork", "swap_out") and model.swapped.get(op[1]):
            continue
        if kind == "swap_in" and not model.swapped.get(op[1]):
            continue
        res = {}
        for name, side in (("m", model), ("p", prod)):
            try:
                if kind == "allocate_cached":
                    res[name] = side.allocate_cached(op[1], op[2])
                elif kind == "append_slot":
                    res[name] = side.append_slot(op[1])
                elif kind == "fork":
                    side.fork(op[1], op[2]); res[name] = "ok"
                elif kind == "swap_out":
                    res[name] = side.swap_out(op[1])
                elif kind == "swap_in":
                    res[name] = side.swap_in(op[1])
                else:
                    side.free(op[1]); res[name] = "ok"
            except (NoBlocks, NoBlocksError):
                res[name] = "noblocks"
            except PkvError:
                res[name] = "invalid"
        assert res["m"] == res["p"], op
        if kind == "allocate_cached" and res["p"] != "noblocks":
            live.add(op[1])
            hits += res["p"] > 0
        elif kind == "fork" and res["p"] == "ok":
            live.add(op[2])
        elif kind == "free":
            live.discard(op[1])
        assert prod.free_queue() == list(model.free_queue)
    assert hits > 20                                     # the workload does hit the cache
    assert [prod.ref_cnt(b) for b in range(nb)] == model.ref_cnt
    assert [prod.block_hash(b) for b in range(nb)] == [model.block_hash(b) for b in range(nb)]
    assert prod.num_cached() == len(model.cached)
    seqs = sorted(s for s in live if not model.swapped.get(s))
    assert prod.export(seqs, 64) == model.export(seqs, 64)


def _reuse_after_different_parent(bm):
    """Two prompts whose second blocks hold the same tokens after different first blocks."""
    a = [1, 2, 3, 4] + [9, 9, 9, 9]
    b = [5, 6, 7, 8] + [9, 9, 9, 9]
    assert bm.allocate_cached(0, a) == 0
    return bm.allocate_cached(1, b)


@pytest.mark.parametrize("side", sorted(MANAGERS))
def test_a_block_is_named_by_its_whole_prefix(side):
    """§3.4: a block's name covers every token before it (the parent's hash), so equal tokens
    after a different parent are not a hit."""
    assert _reuse_after_different_parent(MANAGERS[side](8, 4)) == 0


def test_planted_per_block_key_is_caught():
    """An oracle that named a block by its own tokens only would reuse the second block above."""
    class PerBlockKey(BlockManagerModel):
        def allocate_cached(self, seq, tokens):
            bs = self.block_size
            tokens = [int(t) for t in tokens]
            n_full, need = len(tokens) // bs, -(-len(tokens) // bs)
            hits, table = 0, []
            for i in range(need):
                key = tuple(tokens[i * bs:(i + 1) * bs])
                b = self.cached.get(key) if i < n_full else None
                if b is not None:
                    if self.ref_cnt[b] == 0:
                        self.free_queue.remove(b)
                    self.ref_cnt[b] += 1
                    hits += 1
                else:
                    b = self._pop()
                    if i < n_full:
                        self.cached[key] = b
                        self.block_key[b] = key
                table.append(b)
            self.tables[seq] = table
            self.num_tokens[seq] = len(tokens)
            return hits * bs
    assert _reuse_after_different_parent(PerBlockKey(8, 4)) != 0
