"""The C-ABI library loads, exports every declared symbol, and its host block
manager agrees exactly with the oracle's naive model (CPU only: no kernel is
launched here)."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle.block_manager import BlockManagerError, NaiveBlockManager

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_253_gb300 import build
    build.build()
    from paged_kv_cache_253_gb300 import _lib
    return _lib


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pa_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in sorted(names):
        assert hasattr(so, n), n
    assert names == set(lib.SIGNATURES), "binding and header list the same calls"


def test_error_strings(lib):
    assert lib.pa_error_string(0) == b"ok"
    for code in range(-12, 0):
        assert lib.pa_error_string(code) != b"unknown error"


def test_host_argument_checks_need_no_gpu(lib):
    out = ctypes.c_void_p()
    assert lib.pa_pool_create(0, 16, 8, 128, 1, ctypes.byref(out)) == lib.PA_ERR_INVALID_ARG
    assert lib.pa_pool_create(4, 16, 8, 128, 7, ctypes.byref(out)) == lib.PA_ERR_DTYPE
    assert lib.pa_append_kv(None, None, None, None, 0, None) == lib.PA_ERR_INVALID_ARG
    assert lib.pa_decode(None, None, 1, 8, None, 1, None, 1.0, None, 0, None) == \
        lib.PA_ERR_INVALID_ARG
    assert lib.pa_prefill(None, None, 4, 8, None, 1, 4, None, 1, None, 1.0, None, 0, None) == \
        lib.PA_ERR_INVALID_ARG
    assert lib.pa_pool_set_kv_scales(None, 1.0, 1.0) == lib.PA_ERR_INVALID_ARG
    assert lib.pa_pool_kv_scales(None, None, None) == lib.PA_ERR_INVALID_ARG
    v = ctypes.c_int()
    assert lib.pa_pool_set_option(None, lib.PA_OPT_PARTITION_CAP, 0) == lib.PA_ERR_INVALID_ARG
    assert lib.pa_pool_get_option(None, lib.PA_OPT_PARTITION_CAP, ctypes.byref(v)) == \
        lib.PA_ERR_INVALID_ARG
    assert lib.PA_FP8E4M3 == 2


def test_fnv_vectors(lib):
    from paged_kv_cache_253_gb300.api import fnv1a64
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8




def _compare(cbm, nbm, live):
    assert cbm.free_list() == list(nbm.free)
    assert cbm.evictable_list() == list(nbm.evictable)
    assert cbm.num_evictable() == len(nbm.evictable)
    assert [cbm.refcount(b) for b in range(nbm.num_blocks)] == nbm.refcount
    assert [cbm.is_cached(b) for b in range(nbm.num_blocks)] == \
        [nbm.is_cached(b) for b in range(nbm.num_blocks)]
    for r in live:
        assert cbm.block_table(r) == nbm.block_table(r)
        assert cbm.seq_len(r) == nbm.seq_len(r)


@pytest.mark.parametrize("retain", [False, True], ids=["free-on-release", "retain-evict"])
def test_cpp_block_manager_matches_naive_model(lib, retain):
    from paged_kv_cache_253_gb300.api import BlockManager
    from paged_kv_cache_253_gb300._lib import PagedAttnError
    rng = np.random.default_rng(253 + int(retain))
    for trial in range(40):
        B = int(rng.integers(1, 6))
        nb = int(rng.integers(3, 40))
        order = rng.permutation(nb)
        cbm, nbm = BlockManager(nb, B, order), NaiveBlockManager(nb, B, order, retain=retain)
        cbm.set_retention(retain)
        live = []
        for step in range(250):
            op = int(rng.integers(0, 13))
            if op == 12:
                if retain and rng.random() < 0.2:      # now and then switch retention off and on
                    on = not nbm.retain
                    cbm.set_retention(on)
                    nbm.set_retention(on)
                continue
            if op == 0 or not live:
                toks = rng.integers(0, 3, size=int(rng.integers(0, 3 * B + 1))).tolist()
                salt = int(rng.integers(0, 2))
                a = cbm.add_request(toks, salt)
                b = nbm.add_request(toks, salt)
                assert a == b
                live.append(a[0])
            elif op == 1:
                r = live[int(rng.integers(len(live)))]
                assert cbm.fork(r) == nbm.fork(r)
                live.append(nbm.next_id - 1)
            elif op == 2:
                r = live.pop(int(rng.integers(len(live))))
                cbm.free_request(r)
                nbm.free_request(r)
            elif op == 3:
                reqs = [live[int(i)] for i in rng.integers(0, len(live), size=int(rng.integers(1, 6)))]
                toks = rng.integers(0, 3, size=len(reqs)).tolist()
                exp_slots, exp_pairs, err = [], [], None
                for r, t in zip(reqs, toks):
                    try:
                        s, a, b = nbm.append_slot(r, t)
                    except BlockManagerError:
                        err = True
                        break
                    exp_slots.append(s)
                    if a >= 0:
                        exp_pairs.append((a, b))
                if err:
                    with pytest.raises(PagedAttnError):
                        cbm.append_slots(reqs, toks)
                    # apply the same prefix of entries to the C++ side is what it did
                else:
                    slots, pairs = cbm.append_slots(reqs, toks)
                    assert slots.tolist() == exp_slots
                    assert [tuple(p) for p in pairs.tolist()] == exp_pairs
            else:
                r = live[int(rng.integers(len(live)))]
                t = int(rng.integers(0, 3))
                try:
                    exp = nbm.append_slot(r, t)
                except BlockManagerError:
                    with pytest.raises(PagedAttnError):
                        cbm.append_slot(r, t)
                    continue
                assert cbm.append_slot(r, t) == exp
            _compare(cbm, nbm, live)


def test_batch_tables_and_errors(lib):
    from paged_kv_cache_253_gb300.api import BlockManager
    from paged_kv_cache_253_gb300._lib import PagedAttnError
    bm = BlockManager(6, 4, [3, 1, 4, 0, 5, 2])
    a, _ = bm.add_request([])
    for t in range(9):
        bm.append_slot(a, t)
    b, _ = bm.add_request([])
    bm.append_slot(b, 1)
    tables, lens = bm.batch_tables([a, b])
    assert tables.tolist() == [[3, 1, 4], [0, -1, -1]] and lens.tolist() == [9, 1]
    # the batch's widest table, from one call: 3 blocks for a, 1 for b
    req = np.array([b, a], dtype=np.int32)
    w = ctypes.c_int(-7)
    assert lib.pa_bm_batch_width(bm.handle, 2, req.ctypes.data_as(lib.c_i32p), ctypes.byref(w)) == 0
    assert w.value == 3
    assert lib.pa_bm_batch_width(bm.handle, 1, req.ctypes.data_as(lib.c_i32p), ctypes.byref(w)) == 0
    assert w.value == 1
    assert lib.pa_bm_batch_width(bm.handle, 0, None, ctypes.byref(w)) == 0 and w.value == 0
    bad = np.array([a, 99], dtype=np.int32)
    assert lib.pa_bm_batch_width(bm.handle, 2, bad.ctypes.data_as(lib.c_i32p),
                                 ctypes.byref(w)) == lib.PA_ERR_UNKNOWN_REQUEST
    assert w.value == 0                      # unchanged on error
    assert lib.pa_bm_batch_width(bm.handle, -1, None, ctypes.byref(w)) == lib.PA_ERR_INVALID_ARG
    tables, _ = bm.batch_tables([b])         # width from the batch: one column
    assert tables.tolist() == [[0]]
    with pytest.raises(PagedAttnError):
        bm.free_request(99)
    for t in range(11):                      # b fills the last two free blocks
        bm.append_slot(b, t)
    with pytest.raises(PagedAttnError) as e:
        bm.append_slot(b, 0)
    assert e.value.code == lib.PA_ERR_NO_FREE_BLOCK
    assert bm.seq_len(b) == 12 and bm.num_free() == 0


def test_prefix_groups_follow_the_tables(lib):
    from paged_kv_cache_253_gb300.api import BlockManager
    B = 4
    bm = BlockManager(64, B)
    root, _ = bm.add_request([])
    for t in range(11):                       # 2 full blocks + 3 tokens
        bm.append_slot(root, t)
    kids = [bm.fork(root) for _ in range(3)]
    other, _ = bm.add_request([])
    for t in range(9):
        bm.append_slot(other, t)
    batch = [kids[0], other, root, kids[1], kids[2]]
    for r in batch:                           # each diverges: the partial block is copied
        bm.append_slot(r, 99)
    offs, seqs, nsh = bm.prefix_groups(batch)
    assert offs.tolist() == [0, 4] and seqs.tolist() == [0, 2, 3, 4] and nsh.tolist() == [2]
    tables = [bm.block_table(r) for r in batch]
    for i in seqs.tolist():
        assert tables[i][:2] == tables[0][:2]
    assert len({tables[i][2] for i in seqs.tolist()}) == 4
    # no sharing at all: no groups
    offs, seqs, nsh = bm.prefix_groups([other])
    assert offs.tolist() == [0] and len(nsh) == 0


def test_retention_evicts_and_reuses_in_the_cpp_manager(lib):
    """Once the free pool is empty a retained block is evicted and reused: the
    new owner's appends overwrite it, and a later admission of the old prompt
    no longer hits it."""
    from paged_kv_cache_253_gb300.api import BlockManager
    B, nb = 16, 4
    bm = BlockManager(nb, B)
    bm.set_retention(True)
    a, _ = bm.add_request([])
    for t in range(2 * B):
        bm.append_slot(a, t)
    bm.free_request(a)
    assert bm.evictable_list() == [1, 0]
    c, _ = bm.add_request([])
    for t in range(2 * B + 1):                        # blocks 2, 3, then evicts block 1
        bm.append_slot(c, 100 + t)
    assert bm.block_table(c) == [2, 3, 1] and not bm.is_cached(1)
    d, cached = bm.add_request(list(range(2 * B)))
    assert cached == B and bm.block_table(d) == [0]    # block 0 still hits, block 1 does not
