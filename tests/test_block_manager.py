"""The host block manager (include/wf_blocks.h) on the CPU: a plain Python model of
the documented rules (ember "The core idea": position p in block table[p // P] at
p % P; tiny-vllm-py "Mental Model" and "Prefix Sharing": blocks handed out as a
request grows, shared prefixes with copy-on-write of a shared partial block)
driven with the native manager through random operation sequences."""
import numpy as np
import pytest

from paged_kv_cache_wf_gb300 import binding as wf
from paged_kv_cache_wf_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    wf.load()


class Model:
    """The documented behaviour, written out plainly."""

    def __init__(self, N, P, order):
        self.N, self.P = N, P
        self.free = list(reversed(order))      # pop() takes the next block
        self.ref = [0] * N
        self.seqs = {}                         # id -> [blocks, len]

    def _take(self):
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def _drop(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def append(self, seq, n):
        blocks, length = self.seqs.get(seq, [[], 0])
        cow = n > 0 and seq in self.seqs and length % self.P != 0 and self.ref[blocks[-1]] > 1
        need = int(cow) + -(-(length + n) // self.P) - -(-length // self.P)
        if need > len(self.free):
            return None
        blocks = list(blocks)
        pair = None
        if cow:
            src, dst = blocks[-1], self._take()
            self._drop(src)
            blocks[-1] = dst
            pair = (src, dst)
        slots = []
        for i in range(n):
            pos = length + i
            if pos % self.P == 0:
                blocks.append(self._take())
            slots.append(blocks[pos // self.P] * self.P + pos % self.P)
        self.seqs[seq] = [blocks, length + n]
        return slots, pair

    def fork(self, parent, child):
        blocks, length = self.seqs[parent]
        for b in blocks:
            self.ref[b] += 1
        self.seqs[child] = [list(blocks), length]

    def free_seq(self, seq):
        blocks, _ = self.seqs.pop(seq)
        for b in reversed(blocks):
            self._drop(b)


def _same_state(bm, model):
    assert bm.num_free() == len(model.free)
    assert [bm.ref_count(b) for b in range(model.N)] == model.ref
    for s, (blocks, length) in model.seqs.items():
        assert bm.seq_len(s) == length
        bt, sl = bm.tables([s], max(len(blocks), 1), -7)
        assert list(bt[0][:len(blocks)]) == blocks and int(sl[0]) == length


def test_fresh_manager_hands_out_blocks_in_order_and_slots_follow_the_table():
    bm = wf.BlockManager(8, 4)
    slots, pair = bm.append(11, 6)
    assert pair is None and list(slots) == [0, 1, 2, 3, 4, 5]          # blocks 0 then 1
    slots, _ = bm.append(12, 3)
    assert list(slots) == [8, 9, 10]                                    # block 2
    slots, _ = bm.append(11, 3)
    assert list(slots) == [6, 7, 12]                                    # rest of block 1, then block 3
    bt, sl = bm.tables([11, 12], 4, -1)
    assert bt.tolist() == [[0, 1, 3, -1], [2, -1, -1, -1]] and sl.tolist() == [9, 3]
    assert bm.num_free() == 4 and bm.seq_len(99) == -1


def test_shuffled_free_list_is_a_seeded_permutation():
    a, b, c = wf.BlockManager(64, 16, 5), wf.BlockManager(64, 16, 5), wf.BlockManager(64, 16, 6)
    sa = a.append(1, 64 * 16)[0] // 16
    sb = b.append(1, 64 * 16)[0] // 16
    sc = c.append(1, 64 * 16)[0] // 16
    order_a = list(dict.fromkeys(sa.tolist()))
    assert sorted(order_a) == list(range(64)) and order_a != list(range(64))
    assert np.array_equal(sa, sb) and not np.array_equal(sa, sc)


def test_out_of_blocks_changes_nothing():
    bm = wf.BlockManager(3, 4)
    bm.append(1, 9)                                                     # 3 blocks
    before = (bm.num_free(), [bm.ref_count(b) for b in range(3)], bm.seq_len(1))
    with pytest.raises(wf.WfError) as e:
        bm.append(1, 4)
    assert e.value.code == wf.WF_ERR_NO_BLOCKS
    assert (bm.num_free(), [bm.ref_count(b) for b in range(3)], bm.seq_len(1)) == before
    slots, _ = bm.append(1, 3)                                          # still fits the last block
    assert list(slots) == [9, 10, 11]


def test_prefix_sharing_copies_a_shared_partial_block_once():
    bm = wf.BlockManager(10, 4)
    bm.append(1, 6)                                                     # blocks 0, 1 (1 half full)
    bm.fork(1, 2)
    assert bm.ref_count(0) == 2 and bm.ref_count(1) == 2
    slots, pair = bm.append(2, 1)                                       # 2 writes into shared block 1
    assert pair == (1, 2) and list(slots) == [2 * 4 + 2]
    assert bm.ref_count(1) == 1 and bm.ref_count(2) == 1 and bm.ref_count(0) == 2
    slots, pair = bm.append(1, 1)                                       # 1 now owns block 1 alone
    assert pair is None and list(slots) == [1 * 4 + 2]
    bm.fork(1, 3)
    bm.append(1, 1)                                                     # fills block 1 (shared) -> copy
    bm.free(3)
    bm.free(2)
    bm.free(1)
    assert bm.num_free() == 10 and all(bm.ref_count(b) == 0 for b in range(10))


def test_fork_of_a_full_tail_needs_no_copy_and_bad_ids_are_rejected():
    bm = wf.BlockManager(6, 4)
    bm.append(1, 8)
    bm.fork(1, 2)
    slots, pair = bm.append(2, 2)
    assert pair is None and list(slots) == [8, 9]                       # a new block 2
    for call in (lambda: bm.fork(1, 2), lambda: bm.fork(7, 8), lambda: bm.free(7),
                 lambda: bm.tables([1, 7], 4, 0), lambda: bm.tables([1], 1, 0)):
        with pytest.raises(wf.WfError) as e:
            call()
        assert e.value.code == wf.WF_ERR_INVALID_ARG


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_churn_matches_the_model(seed):
    """Arrivals, growth by one or many tokens, forks, frees and pool exhaustion in
    random order; the native manager and the model agree on every slot, copy pair,
    reference count and table, and no two live sequences share a slot outside a
    shared block."""
    rng = np.random.default_rng(seed)
    N, P = 40, 8
    shuffle = 1000 + seed
    bm = wf.BlockManager(N, P, shuffle)
    order = list(dict.fromkeys((wf.BlockManager(N, P, shuffle).append(0, N * P)[0] // P).tolist()))
    model = Model(N, P, order)
    next_id = 0
    for _ in range(600):
        live = list(model.seqs)
        op = rng.choice(["new", "grow", "grow", "grow", "fork", "free"])
        if op == "new" or not live:
            n = int(rng.integers(0, 3 * P))
            seq = next_id
            next_id += 1
        elif op == "fork":
            parent = int(rng.choice(live))
            child = next_id
            next_id += 1
            bm.fork(parent, child)
            model.fork(parent, child)
            _same_state(bm, model)
            continue
        elif op == "free":
            seq = int(rng.choice(live))
            bm.free(seq)
            model.free_seq(seq)
            _same_state(bm, model)
            continue
        else:
            seq = int(rng.choice(live))
            n = int(rng.integers(1, 2 * P)) if rng.random() < 0.3 else 1
        want = model.append(seq, n)
        if want is None:
            with pytest.raises(wf.WfError):
                bm.append(seq, n)
        else:
            slots, pair = bm.append(seq, n)
            assert list(slots) == want[0] and pair == want[1]
        _same_state(bm, model)
        # slot ownership: a block is in several tables only while shared
        owners = {}
        for s, (blocks, _) in model.seqs.items():
            for b in blocks:
                owners.setdefault(b, set()).add(s)
        for b, who in owners.items():
            assert len(who) == model.ref[b]
