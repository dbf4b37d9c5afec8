"""The decode's split of work over worker warps, and the facts the split-KV merge relies on.

The decode kernel flattens the units of every (sequence, kv head) segment (16-row tiles, or
partitions of part_blocks tiles) and gives worker w the units from floor(w * units / W) up
to the next worker's start.  The merge kernel never reads anything the decode kernel writes
about this split: it works out each segment's pieces from the lengths with two closed
forms, checked here against the definition by brute force:

* the worker of unit u is floor(((u + 1) W - 1) / units);
* worker w's range starts at floor(w * units / W);

and the slot rule.  A piece that covers its whole segment is finished by the decode kernel
itself and takes no slot.  Any other piece takes one of its worker's two slots: 2w if it
starts the worker's range, else 2w + 1.  A range holds at most one piece of the second kind,
the one that starts inside the range and runs past its end.
"""
import random


def start_of(w, units, W):
    return w * units // W


def worker_of(u, units, W):
    return ((u + 1) * W - 1) // units


def segments_units(lens, num_kv_heads, part_blocks):
    """Units per segment, in the decode's flattened order (sequence-major, kv head minor)."""
    out = []
    for L in lens:
        nb = (L + 15) // 16
        nu = (nb + part_blocks - 1) // part_blocks if part_blocks else nb
        out += [nu] * num_kv_heads
    return out


def test_worker_of_unit_is_the_last_worker_starting_at_or_before_it():
    rng = random.Random(160)
    for _ in range(400):
        units = rng.randint(1, 6000)
        W = rng.randint(1, min(units, 2000))
        starts = [start_of(w, units, W) for w in range(W + 1)]
        assert starts[0] == 0 and starts[W] == units
        assert all(starts[w] <= starts[w + 1] for w in range(W))
        for u in rng.sample(range(units), min(units, 60)) + [0, units - 1]:
            brute = max(w for w in range(W) if starts[w] <= u)
            assert worker_of(u, units, W) == brute, (units, W, u)


def test_pieces_slots_and_the_merge_descriptor():
    rng = random.Random(161)
    for _ in range(150):
        S = rng.randint(1, 80)
        hkv = rng.randint(1, 8)
        pb = rng.choice([0, 0, 1, 4, 32])
        lens = [rng.choice([0, rng.randint(1, 40), rng.randint(1, 3000)]) for _ in range(S)]
        seg_units = segments_units(lens, hkv, pb)
        units = sum(seg_units)
        if units == 0:
            continue
        W = min(rng.randint(1, 2000), units)
        starts = [start_of(w, units, W) for w in range(W + 1)]
        # Brute force: walk every worker's range and cut it into pieces at segment ends.
        slots_used = {}
        first_piece = {}
        pieces = {}
        seg_first = []
        acc = 0
        for n in seg_units:
            seg_first.append(acc)
            acc += n
        seg_of_unit = []
        for sidx, n in enumerate(seg_units):
            seg_of_unit += [sidx] * n
        for w in range(W):
            u = starts[w]
            while u < starts[w + 1]:
                sidx = seg_of_unit[u]
                seg_end = seg_first[sidx] + seg_units[sidx]
                end = min(starts[w + 1], seg_end)
                pieces.setdefault(sidx, []).append(w)
                complete = u == seg_first[sidx] and end == seg_end
                if not complete:
                    slot = 2 * w + (0 if u == starts[w] else 1)
                    assert slot not in slots_used, "two partial pieces in one slot"
                    slots_used[slot] = sidx
                    if u != starts[w]:
                        assert end == starts[w + 1], "a partial piece inside the range must run past its end"
                    if u == seg_first[sidx]:
                        first_piece[sidx] = (w, slot)
                u = end
        # The merge's closed forms give the same workers, count and first slot.
        for sidx, n in enumerate(seg_units):
            if n == 0:
                assert sidx not in pieces
                continue
            u0, u1 = seg_first[sidx], seg_first[sidx] + n - 1
            w0 = worker_of(u0, units, W)
            np_ = worker_of(u1, units, W) - w0 + 1
            z = 0 if start_of(w0, units, W) == u0 else 1
            assert pieces[sidx] == list(range(w0, w0 + np_)), (sidx, pieces[sidx], w0, np_)
            if np_ == 1:
                assert sidx not in first_piece             # finished by the decode kernel: no slot
                continue
            assert first_piece[sidx] == (w0, 2 * w0 + z)
            # every later piece starts its worker's range: slot 2w
            for w in range(w0 + 1, w0 + np_):
                assert slots_used[2 * w] == sidx
