"""Pins for the oracle's data movement and naive block manager (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import kvcache as okv
from oracle.block_manager import (BlockManagerError, NaiveBlockManager, block_hash,
                                  fnv1a64)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _invariants(bm):
    refs = [0] * bm.num_blocks
    for req in bm.requests.values():
        for b in req["table"]:
            refs[b] += 1
    assert refs == bm.refcount
    free = list(bm.free)
    assert len(set(free)) == len(free)
    assert not (set(free) & set(bm.evictable)) and len(set(bm.evictable)) == len(bm.evictable)
    for b in range(bm.num_blocks):
        # a block nobody holds is either free or (retention) cached and evictable
        assert (b in set(free) or b in set(bm.evictable)) == (bm.refcount[b] == 0)
    for b in bm.evictable:
        assert b in bm.block_key
    for req in bm.requests.values():
        n = len(req["tokens"])
        slots = len(req["table"]) * bm.block_size
        assert 0 <= slots - n <= bm.block_size - 1        # tail waste below one block
    for h, (blk, _, _) in bm.cache.items():
        assert bm.block_key[blk] == h and (bm.refcount[blk] > 0 or blk in bm.evictable)


# -- data movement --------------------------------------------------------
def test_append_writes_the_worked_example_slot_only():
    g = _golden("worked_address.json")
    B, nb, hkv, D = g["block_size"], 16, 2, 8
    K = np.zeros((nb, hkv, B, D), np.float32)
    V = np.zeros_like(K)
    slot = okv.slot_of(g["token_position"], B, g["block_table"])
    assert slot == g["physical_block"] * B + g["offset"]
    k = np.arange(hkv * D, dtype=np.float32).reshape(1, hkv, D) + 1
    okv.append_kv(K, V, k, -k, [slot])
    assert np.array_equal(K[g["physical_block"], :, g["offset"], :], k[0])
    assert np.array_equal(V[g["physical_block"], :, g["offset"], :], -k[0])
    K[g["physical_block"], :, g["offset"], :] = 0
    V[g["physical_block"], :, g["offset"], :] = 0
    assert not K.any() and not V.any()


def test_negative_slot_is_skipped_and_out_of_pool_rejected():
    K = np.zeros((4, 1, 4, 2), np.uint16)
    V = np.zeros_like(K)
    okv.append_kv(K, V, np.ones((1, 1, 2), np.uint16), np.ones((1, 1, 2), np.uint16), [-1])
    assert not K.any()
    with pytest.raises(ValueError):
        okv.append_kv(K, V, np.ones((1, 1, 2), np.uint16), np.ones((1, 1, 2), np.uint16), [16])


def test_copy_blocks_is_a_bitwise_whole_block_copy():
    rng = np.random.default_rng(0)
    K = rng.integers(0, 1 << 16, size=(8, 2, 4, 3), dtype=np.uint16)
    V = rng.integers(0, 1 << 16, size=(8, 2, 4, 3), dtype=np.uint16)
    K0, V0 = K.copy(), V.copy()
    okv.copy_blocks(K, V, [(1, 6), (3, 0)])
    assert np.array_equal(K[6], K0[1]) and np.array_equal(V[6], V0[1])
    assert np.array_equal(K[0], K0[3]) and np.array_equal(V[0], V0[3])
    untouched = [b for b in range(8) if b not in (0, 6)]
    assert np.array_equal(K[untouched], K0[untouched])
    assert np.array_equal(V[untouched], V0[untouched])


# -- block manager --------------------------------------------------------
def test_growth_example():
    g = _golden("growth.json")
    B = g["block_size"]
    bm = NaiveBlockManager(8, B)
    rid, cached = bm.add_request([])
    assert cached == 0
    for t in range(g["tokens"]):
        bm.append_slot(rid, t)
    assert len(bm.block_table(rid)) == g["blocks"]
    assert len(bm.block_table(rid)) * B - bm.seq_len(rid) == g["unused_slots"]
    free_before = bm.num_free()
    for t in g["tokens_without_new_block"]:
        bm.append_slot(rid, t)
        assert bm.num_free() == free_before
    assert bm.seq_len(rid) == g["token_needing_fourth_block"] - 1
    bm.append_slot(rid, 99)
    assert len(bm.block_table(rid)) == 4 and bm.num_free() == free_before - 1
    _invariants(bm)


def test_free_pool_is_fifo_in_given_order():
    bm = NaiveBlockManager(5, 2, free_order=[3, 1, 4, 0, 2])
    r, _ = bm.add_request([])
    for t in range(5):
        bm.append_slot(r, t)
    assert bm.block_table(r) == [3, 1, 4]
    bm.free_request(r)
    assert list(bm.free) == [0, 2, 3, 1, 4]


def test_slot_encoding_matches_translation():
    bm = NaiveBlockManager(16, 4, free_order=list(np.random.default_rng(3).permutation(16)))
    r, _ = bm.add_request([])
    slots = [bm.append_slot(r, t)[0] for t in range(11)]
    table = bm.block_table(r)
    assert slots == [okv.slot_of(p, 4, table) for p in range(11)]


def test_refcount_lifetime():
    bm = NaiveBlockManager(8, 4)
    a, _ = bm.add_request([])
    for t in range(6):
        bm.append_slot(a, t)
    b = bm.fork(a)
    blocks = bm.block_table(a)
    assert all(bm.refcount[x] == 2 for x in blocks)
    bm.free_request(b)                        # one user leaves: nothing is freed
    assert all(bm.refcount[x] == 1 for x in blocks)
    assert not set(blocks) & set(bm.free)
    bm.free_request(a)                        # the last user leaves
    assert set(blocks) <= set(bm.free)
    _invariants(bm)
    with pytest.raises(BlockManagerError):
        bm.free_request(a)


def test_copy_on_write_repoints_only_the_writer():
    bm = NaiveBlockManager(8, 4, free_order=[5, 2, 7, 0, 1, 3, 4, 6])
    a, _ = bm.add_request([])
    for t in range(6):
        bm.append_slot(a, t)
    assert bm.block_table(a) == [5, 2]
    b = bm.fork(a)
    slot, src, dst = bm.append_slot(b, 100)
    assert (src, dst) == (2, 7)
    assert bm.block_table(b) == [5, 7] and bm.block_table(a) == [5, 2]
    assert slot == 7 * 4 + 2
    assert bm.refcount[5] == 2 and bm.refcount[2] == 1 and bm.refcount[7] == 1
    slot, src, dst = bm.append_slot(a, 200)   # sole owner now: in place
    assert (src, dst) == (-1, -1) and slot == 2 * 4 + 2
    _invariants(bm)


def test_full_shared_blocks_are_never_copied():
    bm = NaiveBlockManager(64, 4)
    a, _ = bm.add_request([])
    for t in range(8):                        # two full blocks
        bm.append_slot(a, t)
    kids = [bm.fork(a) for _ in range(5)]
    pairs = [bm.append_slot(r, 1)[1:] for r in [a] + kids]
    assert all(p == (-1, -1) for p in pairs)
    _invariants(bm)


def test_shared_prefix_divergence_count():
    """256 requests share a 4104-token prompt (256 full blocks + one with 8
    tokens, refcount 256); each first divergent write copies the partial block
    except the last one, which finds itself the only user."""
    B, n_req = 16, 256
    bm = NaiveBlockManager(257 + 300, B)
    root, _ = bm.add_request([])
    for t in range(4104):
        bm.append_slot(root, t % 1000)
    kids = [bm.fork(root) for _ in range(n_req - 1)]
    table = bm.block_table(root)
    assert len(table) == 257 and all(bm.refcount[b] == n_req for b in table)
    pairs = []
    for r in [root] + kids:
        _, src, dst = bm.append_slot(r, 7)
        if src >= 0:
            pairs.append((src, dst))
    assert len(pairs) == n_req - 1
    assert all(src == table[-1] for src, _ in pairs)
    assert len({dst for _, dst in pairs}) == n_req - 1
    assert all(bm.refcount[b] == n_req for b in table[:-1])
    assert bm.refcount[table[-1]] == 1
    _invariants(bm)


def test_no_free_block_leaves_state_unchanged():
    bm = NaiveBlockManager(2, 2)
    a, _ = bm.add_request([])
    for t in range(4):
        bm.append_slot(a, t)
    with pytest.raises(BlockManagerError):
        bm.append_slot(a, 4)
    assert bm.seq_len(a) == 4 and bm.block_table(a) == [0, 1]
    b = bm.fork(a)
    bm.free_request(a)
    _invariants(bm)
    assert bm.refcount == [1, 1]


def test_fnv1a64_published_vectors():
    """FNV-1a 64-bit test vectors published with the FNV hash definition
    (Fowler, Noll, Vo; offset basis 0xcbf29ce484222325, prime 2^40 + 0x1b3)."""
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_prefix_cache_hits_follow_the_parent_chain():
    B = 4
    bm = NaiveBlockManager(32, B)
    prompt = list(range(10, 21))               # 11 tokens: 2 full blocks + 3
    a, cached = bm.add_request(prompt)
    assert cached == 0
    for t in prompt:
        bm.append_slot(a, t)
    ta = bm.block_table(a)
    assert bm.is_cached(ta[0]) and bm.is_cached(ta[1]) and not bm.is_cached(ta[2])
    b, cached = bm.add_request(prompt[:9] + [0, 0])
    assert cached == 8 and bm.block_table(b) == ta[:2]
    assert bm.refcount[ta[0]] == 2 and bm.refcount[ta[1]] == 2
    c, cached = bm.add_request(prompt, salt=1)          # different cache key
    assert cached == 0
    d, cached = bm.add_request([99] * 4 + prompt[4:])   # same 2nd block, other parent
    assert cached == 0
    e, cached = bm.add_request(prompt[:4] + [0] * 4)    # first block only
    assert cached == 4
    _invariants(bm)
    # the hash of block 1 depends on block 0's hash, not on its tokens alone
    h0 = block_hash(0, 0, prompt[:4])
    assert block_hash(h0, 0, prompt[4:8]) != block_hash(0, 0, prompt[4:8])


def test_cached_block_leaves_the_table_with_its_last_user():
    bm = NaiveBlockManager(8, 2)
    a, _ = bm.add_request([1, 2, 3])
    for t in [1, 2, 3]:
        bm.append_slot(a, t)
    bm.free_request(a)
    assert not bm.cache and not bm.block_key
    b, cached = bm.add_request([1, 2, 3])
    assert cached == 0


def test_random_operation_sequences_keep_invariants():
    rng = np.random.default_rng(12)
    for trial in range(30):
        B = int(rng.integers(1, 6))
        nb = int(rng.integers(4, 40))
        bm = NaiveBlockManager(nb, B, free_order=list(rng.permutation(nb)))
        live = []
        for step in range(200):
            op = rng.integers(0, 10)
            try:
                if op == 0 or not live:
                    toks = rng.integers(0, 3, size=int(rng.integers(0, 3 * B + 1))).tolist()
                    r, cached = bm.add_request(toks)
                    live.append(r)
                    assert cached % B == 0 and cached <= len(toks)
                elif op == 1:
                    live.append(bm.fork(live[int(rng.integers(len(live)))]))
                elif op == 2:
                    r = live.pop(int(rng.integers(len(live))))
                    bm.free_request(r)
                else:
                    bm.append_slot(live[int(rng.integers(len(live)))], int(rng.integers(0, 3)))
            except BlockManagerError:
                pass
            _invariants(bm)


# -- retention of cached blocks (eviction) ---------------------------------

def _fill(bm, toks):
    r, cached = bm.add_request(toks)
    for t in toks[cached:]:
        bm.append_slot(r, t)
    return r


def test_retention_keeps_a_finished_prefix_for_the_next_request():
    bm = NaiveBlockManager(6, 2, retain=True)
    a = _fill(bm, [1, 2, 3, 4, 5])                 # blocks 0, 1 full, 2 partial
    assert bm.block_table(a) == [0, 1, 2]
    bm.free_request(a)
    assert bm.evictable == [1, 0]                  # deepest first; the partial block is free
    assert list(bm.free) == [3, 4, 5, 2]
    b, cached = bm.add_request([1, 2, 3, 4, 9])
    assert cached == 4 and bm.block_table(b) == [0, 1]
    assert bm.evictable == [] and bm.refcount[:2] == [1, 1]
    assert list(bm.free) == [3, 4, 5, 2]           # nothing was allocated for the hit
    _invariants(bm)


def test_retention_evicts_least_recently_released_leaves_first():
    bm = NaiveBlockManager(4, 2, retain=True)
    a = _fill(bm, [1, 2, 3, 4])                    # blocks 0, 1
    b = _fill(bm, [7, 8, 9, 9])                    # blocks 2, 3
    bm.free_request(a)
    bm.free_request(b)
    assert bm.evictable == [1, 0, 3, 2] and not bm.free
    c = _fill(bm, [5, 5])                          # needs one block: evicts a's last block
    assert bm.block_table(c) == [1]
    assert bm.evictable == [0, 3, 2]
    d, cached = bm.add_request([1, 2, 3, 4])       # a's first block still hits; its second is gone
    assert cached == 2 and bm.block_table(d) == [0]
    _invariants(bm)


def test_retention_evicts_only_when_the_free_pool_is_empty():
    bm = NaiveBlockManager(5, 2, retain=True)
    a = _fill(bm, [1, 2])
    bm.free_request(a)
    assert bm.evictable == [0] and list(bm.free) == [1, 2, 3, 4]
    b = _fill(bm, [6, 6, 6, 6, 6, 6, 6, 6])        # four new blocks: the free pool suffices
    assert bm.block_table(b) == [1, 2, 3, 4] and bm.evictable == [0] and bm.is_cached(0)
    bm.append_slot(b, 6)                           # a fifth block: only the evictable one is left
    assert bm.block_table(b)[-1] == 0 and bm.evictable == []
    assert not bm.is_cached(0)                     # evicted; registered again only once it fills
    _invariants(bm)


def test_turning_retention_off_returns_retained_blocks_to_the_pool():
    bm = NaiveBlockManager(4, 2, retain=True)
    a = _fill(bm, [1, 2, 3, 4])
    bm.free_request(a)
    assert bm.evictable == [1, 0]
    bm.set_retention(False)
    assert bm.evictable == [] and not bm.cache and not bm.block_key
    assert list(bm.free) == [2, 3, 1, 0]
    _invariants(bm)


def test_random_operation_sequences_keep_invariants_with_retention():
    rng = np.random.default_rng(13)
    for trial in range(30):
        B = int(rng.integers(1, 6))
        nb = int(rng.integers(4, 40))
        bm = NaiveBlockManager(nb, B, free_order=list(rng.permutation(nb)), retain=True)
        live = []
        for step in range(200):
            op = rng.integers(0, 12)
            try:
                if op == 0 or not live:
                    toks = rng.integers(0, 3, size=int(rng.integers(0, 3 * B + 1))).tolist()
                    r, cached = bm.add_request(toks)
                    live.append(r)
                    assert cached % B == 0 and cached <= len(toks)
                elif op == 1:
                    live.append(bm.fork(live[int(rng.integers(len(live)))]))
                elif op in (2, 3):
                    r = live.pop(int(rng.integers(len(live))))
                    bm.free_request(r)
                elif op == 4 and rng.random() < 0.1:
                    bm.set_retention(not bm.retain)
                else:
                    bm.append_slot(live[int(rng.integers(len(live)))], int(rng.integers(0, 3)))
            except BlockManagerError:
                pass
            _invariants(bm)
