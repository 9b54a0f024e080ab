"""The host-side block manager (no GPU): free list, reference counts, page tables,
prefix sharing by fork and copy on write on append.  Checked against invariants and
against a small Python model of the same rules."""

import random

import pytest

import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import build

BS = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def test_allocation_order_and_slots():
    m = pkv.BlockManager(num_blocks=8, max_seqs=4, max_blocks_per_seq=4)
    s = m.add_sequence()
    slots, pairs = m.append([s], [20])
    assert len(pairs) == 0
    assert slots.tolist() == list(range(16)) + [16, 17, 18, 19]  # blocks 0 and 1
    bt, cl = m.tables([s])
    assert bt[0].tolist() == [0, 1, -1, -1] and cl.tolist() == [20]
    assert m.stats() == (6, 1)
    assert [m.refcount(b) for b in range(3)] == [1, 1, 0]


def test_fork_shares_and_copy_on_write():
    m = pkv.BlockManager(num_blocks=10, max_seqs=4, max_blocks_per_seq=4)
    p = m.add_sequence()
    m.append([p], [20])                       # blocks 0 (full), 1 (4 tokens)
    c = m.fork(p)
    assert m.refcount(0) == 2 and m.refcount(1) == 2
    slots, pairs = m.append([c], [1])         # child writes into the shared partial block
    assert pairs.tolist() == [[1, 2]]         # copied to a fresh block first
    assert slots.tolist() == [2 * BS + 4]
    assert m.refcount(1) == 1 and m.refcount(2) == 1 and m.refcount(0) == 2
    slots, pairs = m.append([p], [1])         # the parent now owns block 1 alone
    assert pairs.numel() == 0 and slots.tolist() == [1 * BS + 4]
    bt, cl = m.tables([p, c])
    assert bt[:, :2].tolist() == [[0, 1], [0, 2]] and cl.tolist() == [21, 21]
    m.free_sequence(p)
    assert m.refcount(0) == 1 and m.refcount(1) == 0
    m.free_sequence(c)
    assert m.stats() == (10, 0)


def test_full_shared_blocks_stay_shared():
    m = pkv.BlockManager(num_blocks=10, max_seqs=4, max_blocks_per_seq=4)
    p = m.add_sequence()
    m.append([p], [32])                       # two full blocks
    c = m.fork(p)
    slots, pairs = m.append([p, c], [1, 1])   # both start new blocks: no copy needed
    assert pairs.numel() == 0
    assert slots.tolist() == [2 * BS, 3 * BS]
    assert m.refcount(0) == 2 and m.refcount(1) == 2


def test_errors_change_nothing():
    m = pkv.BlockManager(num_blocks=3, max_seqs=2, max_blocks_per_seq=2)
    s = m.add_sequence()
    m.append([s], [16])
    with pytest.raises(pkv.PagedKVError, match="capacity"):
        m.append([s], [17])                   # would need 3 blocks > max_blocks_per_seq
    t = m.add_sequence()
    with pytest.raises(pkv.PagedKVError, match="capacity"):
        m.append([s, t], [16, 17])            # needs 3 free blocks, 2 left
    assert m.stats() == (2, 2) and m.tables([s])[1].tolist() == [16]
    with pytest.raises(pkv.PagedKVError, match="capacity"):
        m.add_sequence()
    with pytest.raises(pkv.PagedKVError, match="invalid"):
        m.append([s, s], [1, 1])              # one entry per sequence
    with pytest.raises(pkv.PagedKVError, match="invalid"):
        m.free_sequence(7)


def test_truncate_drops_rejected_drafts():
    """Append k draft tokens, keep an accepted prefix: blocks past it return to the pool,
    and the next append reuses the freed slots (copying first if the block is shared)."""
    m = pkv.BlockManager(num_blocks=10, max_seqs=4, max_blocks_per_seq=4)
    s = m.add_sequence()
    m.append([s], [14])                        # block 0 holds 14 tokens
    slots, _ = m.append([s], [5])              # 5 drafts: 2 in block 0, 3 in block 1
    assert slots.tolist() == [14, 15, 16, 17, 18]
    m.truncate(s, 15)                          # one draft accepted
    assert m.tables([s])[1].tolist() == [15] and m.refcount(1) == 0 and m.stats()[0] == 9
    slots, _ = m.append([s], [2])
    assert slots.tolist() == [15, 16]          # block 1 comes back from the free list
    c = m.fork(s)                              # both share blocks 0 and 1 (17 tokens)
    m.truncate(c, 10)                          # child keeps block 0 only; block 1 stays with s
    assert m.refcount(0) == 2 and m.refcount(1) == 1
    slots, pairs = m.append([c], [1])          # block 0 is shared and partly filled: copy
    assert pairs.tolist() == [[0, 2]] and slots.tolist() == [2 * BS + 10]
    m.truncate(c, 0)
    assert m.tables([c])[1].tolist() == [0] and m.refcount(2) == 0
    for bad in (-1, 18):
        with pytest.raises(pkv.PagedKVError, match="invalid"):
            m.truncate(s, bad)


def test_release_before_keeps_a_window():
    """Sliding window: blocks wholly behind the window go back to the pool, their table
    entries read -1, positions keep counting, and appends and forks carry on."""
    m = pkv.BlockManager(num_blocks=8, max_seqs=4, max_blocks_per_seq=8)
    s = m.add_sequence()
    m.append([s], [40])                        # blocks 0, 1, 2 (8 tokens in block 2)
    m.release_before(s, 35)                    # blocks 0 and 1 hold only tokens < 32 <= 35
    bt, cl = m.tables([s])
    assert bt[0, :3].tolist() == [-1, -1, 2] and cl.tolist() == [40]
    assert m.refcount(0) == 0 and m.refcount(1) == 0 and m.stats()[0] == 7
    m.release_before(s, 10)                    # nothing more to release
    assert m.stats()[0] == 7
    c = m.fork(s)                              # shares block 2 only
    assert m.refcount(2) == 2
    slots, pairs = m.append([c], [1])          # shared partial block: copy first
    assert pairs.tolist() == [[2, 1]] and slots.tolist() == [1 * BS + 8]
    with pytest.raises(pkv.PagedKVError, match="invalid"):
        m.truncate(s, 20)                      # below the released blocks
    m.truncate(s, 32)                          # every kept block released: next append takes a new one
    slots, _ = m.append([s], [1])
    assert slots.tolist() == [2 * BS] and m.tables([s])[0][0, :3].tolist() == [-1, -1, 2]  # block 2 came back
    for bad in (-1, 42):                       # c holds 41 tokens
        with pytest.raises(pkv.PagedKVError, match="invalid"):
            m.release_before(c, bad)
    m.free_sequence(s)
    m.free_sequence(c)
    assert m.stats() == (8, 0)


class Model:
    """The same rules in plain Python."""

    def __init__(self, nb):
        self.ref = [0] * nb
        self.free = list(range(nb - 1, -1, -1))
        self.seqs = {}

    def take(self):
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def drop(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def append(self, s, k):
        blocks, length, released = self.seqs[s]
        slots, pairs = [], []
        for _ in range(k):
            j, off = divmod(length, BS)
            if off == 0:
                blocks.append(self.take())
            elif self.ref[blocks[j]] > 1:
                src, dst = blocks[j], self.take()
                self.drop(src)
                blocks[j] = dst
                pairs.append([src, dst])
            slots.append(blocks[j] * BS + off)
            length += 1
        self.seqs[s] = (blocks, length, released)
        return slots, pairs


def test_random_operations_match_model():
    rng = random.Random(7)
    nb = 64
    m = pkv.BlockManager(num_blocks=nb, max_seqs=16, max_blocks_per_seq=32)
    model = Model(nb)
    for _ in range(600):
        op = rng.random()
        live = list(model.seqs)
        if op < 0.15 and len(live) < 16:
            s = m.add_sequence()
            model.seqs[s] = ([], 0, 0)
        elif op < 0.3 and live and len(live) < 16:
            p = rng.choice(live)
            c = m.fork(p)
            blocks, length, released = model.seqs[p]
            for b in blocks:
                if b >= 0:
                    model.ref[b] += 1
            model.seqs[c] = (list(blocks), length, released)
        elif op < 0.4 and live:
            s = rng.choice(live)
            m.free_sequence(s)
            for b in model.seqs.pop(s)[0]:
                if b >= 0:
                    model.drop(b)
        elif op < 0.5 and live:
            s = rng.choice(live)
            blocks, length, released = model.seqs[s]
            keep = rng.randint(0, length)
            if keep < released * BS:
                with pytest.raises(pkv.PagedKVError):
                    m.truncate(s, keep)
                continue
            m.truncate(s, keep)
            nkeep = -(-keep // BS)
            for b in reversed(blocks[nkeep:]):
                if b >= 0:
                    model.drop(b)
            model.seqs[s] = (blocks[:nkeep], keep, released)
        elif op < 0.58 and live:
            s = rng.choice(live)
            blocks, length, released = model.seqs[s]
            token = rng.randint(0, length)
            m.release_before(s, token)
            upto = token // BS
            for j in range(released, upto):
                if blocks[j] >= 0:
                    model.drop(blocks[j])
                blocks[j] = -1
            model.seqs[s] = (blocks, length, max(released, upto))
        elif live:
            s = rng.choice(live)
            k = rng.randint(0, 20)
            blocks, length, released = model.seqs[s]
            need = -(-(length + k) // BS) - len(blocks) + (1 if length % BS and k and model.ref[blocks[-1]] > 1 else 0)
            if need > len(model.free) or -(-(length + k) // BS) > 32:
                with pytest.raises(pkv.PagedKVError):
                    m.append([s], [k])
                continue
            slots, pairs = m.append([s], [k])
            ms, mp = model.append(s, k)
            assert slots.tolist() == ms and pairs.tolist() == mp
        # invariants after every operation
        assert m.stats()[0] == len(model.free)
        assert all(m.refcount(b) == model.ref[b] for b in range(nb))
        if model.seqs:
            seqs = sorted(model.seqs)
            bt, cl = m.tables(seqs)
            for i, s in enumerate(seqs):
                blocks, length, _ = model.seqs[s]
                assert cl[i] == length and bt[i, :len(blocks)].tolist() == blocks
