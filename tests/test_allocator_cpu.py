"""The host-side block allocator (include/pkv.h, pkv_allocator_*), on the CPU.

Pinned to the worked trace of the nano-vllm KV-cache post (§3.3.3 / §3.3.5:
a pool of 2234 blocks of 256 tokens, sequence 4 of 406 tokens, sequence 5 of
409 tokens sharing its first block), to the post's may_append boundary table
(§3.3.4), and, over random operation sequences, to a small independent model
of the same rules written here.
"""
from collections import deque

import numpy as np
import pytest

from paged_kv_cache_62_gb300 import build as pkv_build
from paged_kv_cache_62_gb300 import pkv


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    pkv.load()


def table(a, seq, max_blocks=64):
    bt, lens = a.tables([seq], max_blocks)
    row = bt[0].tolist()
    return [b for b in row if b >= 0], int(lens[0])


def test_pages_trace_allocate_share_release():
    """§3.3.3 log: seq 4 (406 tokens) -> [0, 1], 2232 free; seq 5 (409 tokens, first block shared) ->
    [0, 2], block 0 ref_count 2, 2231 free.  §3.3.5 log: freeing seq 4 releases block 1 only (2232 free),
    freeing seq 5 releases block 2 then block 0 (2233, 2234)."""
    a = pkv.BlockAllocator(2234, 256)
    a.add(4, 406)
    assert table(a, 4) == ([0, 1], 406)
    assert a.num_free() == 2232
    a.add(5, 409, parent_id=4, shared_blocks=1)
    assert table(a, 5) == ([0, 2], 409)
    assert a.ref_count(0) == 2 and a.ref_count(1) == 1 and a.ref_count(2) == 1
    assert a.num_free() == 2231
    a.free(4)
    assert a.num_free() == 2232 and a.ref_count(1) == 0 and a.ref_count(0) == 1
    a.free(5)
    assert a.num_free() == 2234 and a.ref_count(0) == 0 and a.ref_count(2) == 0
    # released blocks went to the back of the FIFO in release order (1, then 2, then 0): a sequence
    # taking every block gets the never-used ones first, then 1, 2, 0
    a.add(6, 2234 * 256)
    ids, _ = table(a, 6, 2234)
    assert ids == list(range(3, 2234)) + [1, 2, 0]
    assert a.num_free() == 0


def test_may_append_boundaries():
    """§3.3.4 table (block_size 256): the token that makes the length 257 (513) opens a new block; the
    tokens up to a full block do not."""
    a = pkv.BlockAllocator(8, 256)
    a.add(1, 255)
    assert table(a, 1)[0] == [0]
    assert a.append(1) == (-1, -1)          # length 256: fills block 0
    assert table(a, 1) == ([0], 256)
    assert a.append(1) == (-1, -1)          # length 257: block 1
    assert table(a, 1) == ([0, 1], 257)
    for _ in range(255):
        a.append(1)                          # up to 512
    assert table(a, 1) == ([0, 1], 512)
    a.append(1)                              # 513: block 2
    assert table(a, 1) == ([0, 1, 2], 513)
    assert a.num_free() == 5


def test_copy_on_write_after_fork():
    """Parallel sampling (§2.2): a fork shares every block; the first write into the shared half-full
    last block copies it; the other sequence then owns the original alone and writes in place."""
    a = pkv.BlockAllocator(16, 16)
    a.add(1, 40)                             # blocks 0, 1, 2 (block 2 holds tokens 32..39)
    a.fork(1, 2)
    assert table(a, 2) == ([0, 1, 2], 40)
    assert [a.ref_count(b) for b in (0, 1, 2)] == [2, 2, 2]
    src, dst = a.append(2)                   # token 40 -> shared block 2: copy-on-write
    assert (src, dst) == (2, 3)
    assert table(a, 2) == ([0, 1, 3], 41) and table(a, 1) == ([0, 1, 2], 40)
    assert a.ref_count(2) == 1 and a.ref_count(3) == 1
    assert a.append(1) == (-1, -1)           # sequence 1 owns block 2 alone now
    a.add(3, 48)                             # a full last block
    a.fork(3, 4)
    assert a.append(4) == (-1, -1)           # token 48 opens a fresh block: no copy
    assert table(a, 4)[0][:3] == table(a, 3)[0]


def test_errors_leave_the_allocator_unchanged():
    a = pkv.BlockAllocator(4, 16)
    a.add(1, 48)                                      # 3 blocks
    with pytest.raises(pkv.PkvError) as e:
        a.add(2, 33)                                  # needs 3, 1 free
    assert e.value.status == pkv.EFULL
    assert a.num_free() == 1 and a.num_tokens(2) == -1
    for bad in (lambda: a.add(1, 5),                  # id in use
                lambda: a.add(-1, 5),                 # negative id
                lambda: a.add(3, 20, parent_id=9, shared_blocks=1),   # unknown parent
                lambda: a.add(3, 32, parent_id=1, shared_blocks=2),   # would share the last token's block
                lambda: a.add(3, 80, parent_id=1, shared_blocks=4),   # more than the parent holds
                lambda: a.fork(7, 8), lambda: a.fork(1, 1), lambda: a.append(9), lambda: a.free(9)):
        with pytest.raises(pkv.PkvError) as e:
            bad()
        assert e.value.status == pkv.EINVAL
    assert a.num_free() == 1 and [a.ref_count(b) for b in range(4)] == [1, 1, 1, 0]
    a.fork(1, 2)
    a.add(3, 1)                                       # takes the last free block
    with pytest.raises(pkv.PkvError) as e:
        a.append(2)                                   # token 48 needs a fresh block: none
    assert e.value.status == pkv.EFULL
    assert a.num_tokens(2) == 48 and table(a, 2)[0] == [0, 1, 2]
    with pytest.raises(pkv.PkvError):
        a.tables([1, 2], 2)                           # rows of 3 blocks do not fit
    assert pkv.load().pkv_allocator_create(0, 16) is None
    assert a.ref_count(4) == -1 and a.ref_count(-1) == -1


def test_tables_are_padded_and_carry_lengths():
    a = pkv.BlockAllocator(10, 8)
    a.add(7, 17)
    a.add(3, 1)
    bt, lens = a.tables([3, 7], 4)
    assert bt.tolist() == [[3, -1, -1, -1], [0, 1, 2, -1]]
    assert lens.tolist() == [1, 17]
    with pytest.raises(pkv.PkvError) as e:      # sequence 7 holds 3 blocks: a row of 2 is too short
        a.tables([3, 7], 2)
    assert e.value.status == pkv.EBOUNDS
    with pytest.raises(pkv.PkvError) as e:      # unknown sequence
        a.tables([5], 4)
    assert e.value.status == pkv.EINVAL


class Model:
    """The same rules, written independently for the test: FIFO free list, counts, COW on append."""

    def __init__(self, n, bs):
        self.bs, self.free, self.ref, self.seqs = bs, deque(range(n)), [0] * n, {}

    def take(self):
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def add(self, sid, tokens, parent=-1, shared=0):
        need = -(-tokens // self.bs)
        if sid in self.seqs or sid < 0:
            return pkv.EINVAL
        if shared:
            if parent not in self.seqs or shared > len(self.seqs[parent][1]) or shared * self.bs >= tokens:
                return pkv.EINVAL
        if need - shared > len(self.free):
            return pkv.EFULL
        t = list(self.seqs[parent][1][:shared]) if shared else []
        for b in t:
            self.ref[b] += 1
        while len(t) < need:
            t.append(self.take())
        self.seqs[sid] = [tokens, t]
        return pkv.OK

    def fork(self, p, c):
        if p not in self.seqs or c in self.seqs or c < 0:
            return pkv.EINVAL
        self.seqs[c] = [self.seqs[p][0], list(self.seqs[p][1])]
        for b in self.seqs[c][1]:
            self.ref[b] += 1
        return pkv.OK

    def append(self, sid):
        if sid not in self.seqs:
            return pkv.EINVAL, (-1, -1)
        n, t = self.seqs[sid]
        cow = (-1, -1)
        if n % self.bs == 0:
            if not self.free:
                return pkv.EFULL, cow
            t.append(self.take())
        elif self.ref[t[-1]] > 1:
            if not self.free:
                return pkv.EFULL, cow
            src, dst = t[-1], self.take()
            self.ref[src] -= 1
            t[-1] = dst
            cow = (src, dst)
        self.seqs[sid][0] = n + 1
        return pkv.OK, cow

    def release(self, sid):
        if sid not in self.seqs:
            return pkv.EINVAL
        for b in reversed(self.seqs.pop(sid)[1]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        return pkv.OK


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operations_match_the_model(seed):
    rng = np.random.default_rng(seed)
    NB, bs = 64, 8
    a, m = pkv.BlockAllocator(NB, bs), Model(NB, bs)
    lib = pkv.load()

    def status(fn):
        try:
            fn()
            return pkv.OK
        except pkv.PkvError as e:
            return e.status

    for step in range(3000):
        op = rng.integers(0, 5)
        sid = int(rng.integers(0, 12))
        live = list(m.seqs)
        if op == 0:
            tokens = int(rng.integers(1, 60))
            parent = int(rng.choice(live)) if live and rng.random() < 0.5 else -1
            shared = int(rng.integers(0, 4)) if parent >= 0 else 0
            want = m.add(sid, tokens, parent, shared)
            assert status(lambda: a.add(sid, tokens, parent, shared)) == want, step
        elif op == 1:
            child = int(rng.integers(0, 12))
            want = m.fork(sid, child)
            assert status(lambda: a.fork(sid, child)) == want, step
        elif op in (2, 3):
            want, cow = m.append(sid)
            got = [None]

            def app():
                got[0] = a.append(sid)
            assert status(app) == want, step
            if want == pkv.OK:
                assert got[0] == cow, step
        else:
            want = m.release(sid)
            assert status(lambda: a.free(sid)) == want, step
        # invariants after every step: counts, free list size, tables, lengths
        assert a.num_free() == len(m.free)
        assert [a.ref_count(b) for b in range(NB)] == m.ref
        if m.seqs:
            ids = sorted(m.seqs)
            bt, lens = a.tables(ids, 16)
            for i, s in enumerate(ids):
                n, t = m.seqs[s]
                assert lens[i] == n and [b for b in bt[i].tolist() if b >= 0] == t
        held = sum(len(t) for _, t in m.seqs.values())
        assert sum(m.ref) == held and sum(1 for r in m.ref if r == 0) == len(m.free)
    assert lib.pkv_allocator_num_free(None) == -1


def test_prefix_sharing_tables_of_the_long_mixed_shape():
    """Groups of 8 sequences share up to 64 leading full blocks of the group's first sequence, never
    the block of the last token (the long/mixed workload's structure): shared blocks carry a count of
    (members that share them + 1), every other block 1."""
    rng = np.random.default_rng(4)
    bs, B = 16, 32
    lens = np.exp(rng.uniform(np.log(1), np.log(4096), size=B)).astype(int).clip(1, None)
    need = int(sum(-(-int(L) // bs) for L in lens))
    a = pkv.BlockAllocator(need + 8, bs)
    for g in range(0, B, 8):
        lead = g
        a.add(lead, int(lens[lead]))
        for s in range(g + 1, g + 8):
            # full blocks only: neither sequence's last-token block is shared
            share = min(64, (int(lens[s]) - 1) // bs, (int(lens[lead]) - 1) // bs)
            a.add(s, int(lens[s]), parent_id=lead if share else -1, shared_blocks=share)
    bt, got_lens = a.tables(range(B), 4096 // bs + 1)
    assert got_lens.tolist() == lens.tolist()
    counts = {}
    for row in bt.tolist():
        for b in row:
            if b >= 0:
                counts[b] = counts.get(b, 0) + 1
    assert all(a.ref_count(b) == c for b, c in counts.items())
    # the block holding each sequence's last token is private
    for i, L in enumerate(lens):
        last = bt[i, (int(L) - 1) // bs].item()
        assert a.ref_count(last) == 1, i
