"""Pins for the float64 attention oracle (CPU only).

Each test ties the oracle to something other than itself: the pages' worked
address example, closed forms, torch's float64 scaled-dot-product attention,
and the verification recipe of kgptalkie "Day 28" ("A Tiny Block-Table
Example": the paged output must equal a contiguous computation, whatever the
physical placement of the blocks).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import kvcache as okv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _scatter(k_seq, v_seq, table, B, nb):
    """Place one sequence's contiguous keys/values into a pool through its table,
    using the oracle's append (slots from the pinned translation)."""
    L, hkv, D = k_seq.shape
    K = np.zeros((nb, hkv, B, D), np.float32)
    V = np.zeros_like(K)
    slots = [okv.slot_of(j, B, table) for j in range(L)]
    okv.append_kv(K, V, k_seq, v_seq, slots)
    return K, V


def _random_case(rng, S=3, hq=4, hkv=2, D=16, B=4, max_len=23, nb=40, dtype=np.float32):
    lens = rng.integers(1, max_len + 1, size=S)
    k_seqs = [rng.standard_normal((L, hkv, D)).astype(dtype) for L in lens]
    v_seqs = [rng.standard_normal((L, hkv, D)).astype(dtype) for L in lens]
    perm = rng.permutation(nb)
    width = max(-(-int(L) // B) for L in lens)
    tables = np.full((S, width), -1, np.int32)
    K = np.zeros((nb, hkv, B, D), dtype)
    V = np.zeros_like(K)
    used = 0
    for s, L in enumerate(lens):
        n = -(-int(L) // B)
        tables[s, :n] = perm[used:used + n]
        used += n
        slots = [okv.slot_of(j, B, tables[s]) for j in range(L)]
        okv.append_kv(K, V, k_seqs[s], v_seqs[s], slots)
    q = rng.standard_normal((S, hq, D))
    return q, k_seqs, v_seqs, K, V, tables, lens.astype(np.int32)


def test_worked_address_python_and_c():
    g = _golden("worked_address.json")
    assert okv.translate(g["token_position"], g["block_size"], g["block_table"]) == \
        (g["physical_block"], g["offset"])
    assert divmod(g["token_position"], g["block_size"]) == (g["logical_block"], g["offset"])
    assert oa.translate_c(g["token_position"], g["block_size"], g["block_table"]) == \
        (g["physical_block"], g["offset"])
    # every position of the 9 cached tokens lands in the spans the page lists
    for lb, (lo, hi) in enumerate(g["logical_block_spans"]):
        for p in range(lo, min(hi, g["cached_tokens"] - 1) + 1):
            assert oa.translate_c(p, g["block_size"], g["block_table"])[0] == g["block_table"][lb]


def test_worked_address_inside_attention():
    """The C attention loop reads token 6 from physical block 2, offset 2."""
    g = _golden("worked_address.json")
    B, D, hkv, nb = g["block_size"], 8, 1, 16
    K = np.zeros((nb, hkv, B, D), np.float32)
    V = np.zeros_like(K)
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.0
    K[g["physical_block"], 0, g["offset"], 0] = 50.0 * math.sqrt(D)   # score 50 after scale
    marker = np.arange(1, D + 1, dtype=np.float32)
    V[g["physical_block"], 0, g["offset"], :] = marker
    # a decoy at the transposed address (block 2 of the pool at offset 1 = 6 // 4)
    V[g["block_table"][g["offset"]], 0, g["logical_block"], :] = -100.0
    tables = np.array([g["block_table"]], np.int32)
    out = oa.paged_decode(q, K, V, tables, np.array([7], np.int32), 1.0 / math.sqrt(D), hkv)
    np.testing.assert_allclose(out[0, 0], marker, rtol=0, atol=1e-12)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    q, ks, vs, K, V, tables, _ = _random_case(rng)
    lens = np.ones(len(ks), np.int32)
    out = oa.paged_decode(q, K, V, tables, lens, 0.3, 2)
    for s in range(len(ks)):
        for h in range(q.shape[1]):
            np.testing.assert_array_equal(out[s, h], vs[s][0, h // 2].astype(np.float64))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    L, hkv, D, B = 11, 1, 8, 4
    k_row = rng.standard_normal((1, hkv, D)).astype(np.float32)
    ks = np.repeat(k_row, L, axis=0)
    vs = rng.standard_normal((L, hkv, D)).astype(np.float32)
    table = [5, 0, 3]
    K, V = _scatter(ks, vs, table, B, 8)
    q = rng.standard_normal((1, 1, D))
    out = oa.paged_decode(q, K, V, np.array([table], np.int32), np.array([L], np.int32), 0.7, hkv)
    np.testing.assert_allclose(out[0, 0], vs[:, 0].astype(np.float64).mean(0), rtol=0, atol=1e-14)


def test_zero_length_gives_zeros():
    rng = np.random.default_rng(3)
    q, ks, vs, K, V, tables, lens = _random_case(rng)
    lens[1] = 0
    out = oa.paged_decode(q, K, V, tables, lens, 0.25, 2)
    assert np.all(out[1] == 0.0)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (8, 1), (6, 3)])
def test_matches_torch_sdpa_float64(hq, hkv):
    """Library special case: torch's scaled_dot_product_attention in float64 on
    the contiguous keys, with each KV head repeated for its query-head group."""
    rng = np.random.default_rng(10 + hq * 7 + hkv)
    D = 16
    q, ks, vs, K, V, tables, lens = _random_case(rng, S=4, hq=hq, hkv=hkv, D=D, B=4)
    scale = 1.0 / math.sqrt(D)
    out = oa.paged_decode(q, K, V, tables, lens, scale, hkv)
    for s in range(len(ks)):
        qt = torch.from_numpy(q[s]).unsqueeze(1)                           # [Hq, 1, D]
        kt = torch.from_numpy(ks[s].astype(np.float64)).permute(1, 0, 2)   # [Hkv, L, D]
        vt = torch.from_numpy(vs[s].astype(np.float64)).permute(1, 0, 2)
        kt = kt.repeat_interleave(hq // hkv, dim=0)
        vt = vt.repeat_interleave(hq // hkv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(out[s], ref[:, 0].numpy(), rtol=0, atol=1e-12)


def test_large_scores_stay_finite_and_match_sdpa():
    rng = np.random.default_rng(4)
    q, ks, vs, K, V, tables, lens = _random_case(rng, S=2, hq=2, hkv=2, D=8)
    scale = 400.0
    out = oa.paged_decode(q, K, V, tables, lens, scale, 2)
    assert np.all(np.isfinite(out))
    for s in range(2):
        qt = torch.from_numpy(q[s]).unsqueeze(1)
        kt = torch.from_numpy(ks[s].astype(np.float64)).permute(1, 0, 2)
        vt = torch.from_numpy(vs[s].astype(np.float64)).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(out[s], ref[:, 0].numpy(), rtol=0, atol=1e-10)


def test_paged_equals_contiguous():
    rng = np.random.default_rng(5)
    q, ks, vs, K, V, tables, lens = _random_case(rng, S=5, hq=4, hkv=2, D=8, max_len=30, nb=64)
    paged = oa.paged_decode(q, K, V, tables, lens, 0.35, 2)
    contig = oa.contiguous_decode(q, ks, vs, 0.35, 2)
    np.testing.assert_array_equal(paged, contig)


def test_moving_physical_blocks_leaves_output_unchanged():
    rng = np.random.default_rng(6)
    q, ks, vs, K, V, tables, lens = _random_case(rng, S=4, hq=4, hkv=2, D=8, max_len=30, nb=48)
    base = oa.paged_decode(q, K, V, tables, lens, 0.35, 2)
    for trial in range(3):
        move = rng.permutation(K.shape[0])          # block b moves to move[b]
        K2 = np.empty_like(K)
        V2 = np.empty_like(V)
        K2[move] = K
        V2[move] = V
        t2 = np.where(tables >= 0, move[np.maximum(tables, 0)], -1).astype(np.int32)
        np.testing.assert_array_equal(oa.paged_decode(q, K2, V2, t2, lens, 0.35, 2), base)


def test_sorting_the_table_scrambles_history():
    """Logical order is not physical order: a table sorted by block id reads
    the tokens in a different order.  Decode attention carries no position
    term here, so the change shows where the partly filled last block moves:
    sorted, a different block supplies the unfilled tail."""
    rng = np.random.default_rng(7)
    L, hkv, D, B = 12, 1, 8, 4
    ks = rng.standard_normal((L, hkv, D)).astype(np.float32)
    vs = rng.standard_normal((L, hkv, D)).astype(np.float32)
    table = [14, 9, 2]
    K, V = _scatter(ks, vs, table, B, 16)
    q = rng.standard_normal((1, 1, D))
    lens = np.array([10], np.int32)             # the last block partly filled
    good = oa.paged_decode(q, K, V, np.array([table], np.int32), lens, 0.5, hkv)
    bad = oa.paged_decode(q, K, V, np.array([sorted(table)], np.int32), lens, 0.5, hkv)
    assert np.abs(good - bad).max() > 1e-3


def test_bf16_bits_widen_exactly():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F], np.uint16)
    vals = oa.bf16_bits_to_f32(bits)
    assert vals.tolist()[:5] == [1.0, -2.0, 1.0078125, 0.0, -0.0]
    assert vals[5] == np.float32(3.3895313892515355e38)


def test_bf16_storage_matches_float32_storage():
    """The C loops' bf16 widening gives the same result as passing the exact
    float32 values."""
    rng = np.random.default_rng(8)
    q, ks, vs, K, V, tables, lens = _random_case(rng, S=3, hq=4, hkv=2, D=8)
    Kb = torch.from_numpy(K).to(torch.bfloat16)
    Vb = torch.from_numpy(V).to(torch.bfloat16)
    kbits = Kb.view(torch.int16).numpy().view(np.uint16)
    vbits = Vb.view(torch.int16).numpy().view(np.uint16)
    out_bits = oa.paged_decode(q, kbits, vbits, tables, lens, 0.3, 2)
    out_f32 = oa.paged_decode(q, Kb.float().numpy(), Vb.float().numpy(), tables, lens, 0.3, 2)
    np.testing.assert_array_equal(out_bits, out_f32)


def test_threads_do_not_change_result():
    rng = np.random.default_rng(9)
    q, ks, vs, K, V, tables, lens = _random_case(rng, S=7, hq=4, hkv=2, D=8)
    one = oa.paged_decode(q, K, V, tables, lens, 0.3, 2, threads=1)
    many = oa.paged_decode(q, K, V, tables, lens, 0.3, 2, threads=4)
    np.testing.assert_array_equal(one, many)


def test_bad_block_id_is_reported():
    rng = np.random.default_rng(11)
    q, ks, vs, K, V, tables, lens = _random_case(rng, S=2, hq=2, hkv=2, D=8)
    tables = tables.copy()
    tables[0, 0] = K.shape[0] + 3
    with pytest.raises(ValueError):
        oa.paged_decode(q, K, V, tables, lens, 0.3, 2)
