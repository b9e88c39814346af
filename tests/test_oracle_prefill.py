"""Pins for the paged prefill oracle (CPU only).

The prefill of a whole sequence is causal self-attention, so torch's
scaled_dot_product_attention in float64 with is_causal (grouped heads
expanded) is an independent reference; a chunk must give the same rows as the
whole-sequence prefill (its queries see the cached prefix and the chunk up to
themselves); a fresh sequence's first query returns its own value; a key or
value after a query's position never changes that query's output."""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import prefill as opf


def _pool(rng, lengths, B, hkv, D, extra=3):
    """Random float32 pool, one scattered table per sequence; also the
    contiguous keys/values of each sequence."""
    nb = sum(-(-L // B) for L in lengths) + extra
    k = rng.standard_normal((nb, hkv, B, D)).astype(np.float32)
    v = rng.standard_normal((nb, hkv, B, D)).astype(np.float32)
    order = rng.permutation(nb)
    width = max(1, max(-(-L // B) for L in lengths))
    tables = np.full((len(lengths), width), -1, dtype=np.int32)
    kseq, vseq, o = [], [], 0
    for s, L in enumerate(lengths):
        nbk = -(-L // B)
        tables[s, :nbk] = order[o:o + nbk]
        o += nbk
        blocks = tables[s, :nbk]
        kseq.append(k[blocks].transpose(0, 2, 1, 3).reshape(-1, hkv, D)[:L])
        vseq.append(v[blocks].transpose(0, 2, 1, 3).reshape(-1, hkv, D)[:L])
    return k, v, tables, kseq, vseq


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (6, 2)])
def test_whole_sequence_prefill_matches_sdpa_causal(hq, hkv):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(hq * 10 + hkv)
    B, D = 4, 16
    lengths = [1, 7, 13]
    k, v, tables, kseq, vseq = _pool(rng, lengths, B, hkv, D)
    T = sum(lengths)
    q = rng.standard_normal((T, hq, D))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    scale = 0.37
    out = opf.paged_prefill(q, k, v, tables, cu, np.asarray(lengths, np.int32), scale, hkv)
    G = hq // hkv
    for s, L in enumerate(lengths):
        qs = torch.from_numpy(q[cu[s]:cu[s + 1]]).permute(1, 0, 2)            # [hq, L, D]
        ks = torch.from_numpy(kseq[s].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        vs = torch.from_numpy(vseq[s].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, is_causal=True,
                                                               scale=scale)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_chunks_equal_rows_of_the_whole_prefill():
    rng = np.random.default_rng(5)
    B, hq, hkv, D = 4, 4, 2, 8
    lengths = [11, 20]
    k, v, tables, _, _ = _pool(rng, lengths, B, hkv, D)
    L = np.asarray(lengths, np.int32)
    q_all = rng.standard_normal((sum(lengths), hq, D))
    cu_all = np.array([0, 11, 31], np.int32)
    whole = opf.paged_prefill(q_all, k, v, tables, cu_all, L, 0.5, hkv)
    # chunks: the last 4 tokens of sequence 0, the last 9 of sequence 1
    n = [4, 9]
    rows = np.concatenate([np.arange(11 - 4, 11), 11 + np.arange(20 - 9, 20)])
    cu = np.array([0, 4, 13], np.int32)
    chunk = opf.paged_prefill(q_all[rows], k, v, tables, cu, L, 0.5, hkv)
    np.testing.assert_array_equal(chunk, whole[rows])
    seq, pos = opf.query_positions(cu, L)
    assert seq.tolist() == [0] * 4 + [1] * 9
    assert pos.tolist() == list(range(7, 11)) + list(range(11, 20))
    assert n == np.diff(cu).tolist()


def test_first_query_returns_its_own_value_and_one_token_chunk_is_decode():
    rng = np.random.default_rng(6)
    B, hq, hkv, D = 4, 4, 2, 8
    lengths = [9, 5]
    k, v, tables, kseq, vseq = _pool(rng, lengths, B, hkv, D)
    q = rng.standard_normal((sum(lengths), hq, D))
    cu = np.array([0, 9, 14], np.int32)
    out = opf.paged_prefill(q, k, v, tables, cu, np.asarray(lengths, np.int32), 1.0, hkv)
    G = hq // hkv
    for s in range(2):
        first = out[cu[s]]
        for h in range(hq):
            np.testing.assert_array_equal(first[h], vseq[s][0, h // G].astype(np.float64))
    # a one-token chunk at the end of each context is the decode of that context
    qd = rng.standard_normal((2, hq, D))
    one = opf.paged_prefill(qd, k, v, tables, np.array([0, 1, 2], np.int32),
                            np.asarray(lengths, np.int32), 0.8, hkv)
    dec = oatt.paged_decode(qd, k, v, tables, np.asarray(lengths, np.int32), 0.8, hkv)
    np.testing.assert_array_equal(one, dec)


def test_later_keys_do_not_reach_earlier_queries():
    rng = np.random.default_rng(7)
    B, hq, hkv, D = 4, 2, 1, 8
    lengths = [10]
    k, v, tables, _, _ = _pool(rng, lengths, B, hkv, D, extra=0)
    q = rng.standard_normal((6, hq, D))
    cu = np.array([0, 6], np.int32)                    # positions 4 .. 9
    L = np.asarray(lengths, np.int32)
    before = opf.paged_prefill(q, k, v, tables, cu, L, 1.0, hkv)
    # change the key and value at position 7 (block tables[0][1], offset 3)
    k2, v2 = k.copy(), v.copy()
    b = tables[0][7 // B]
    k2[b, :, 7 % B] += 3.0
    v2[b, :, 7 % B] -= 5.0
    after = opf.paged_prefill(q, k2, v2, tables, cu, L, 1.0, hkv)
    np.testing.assert_array_equal(after[:3], before[:3])          # positions 4, 5, 6
    assert np.all(np.abs(after[3:] - before[3:]).max(axis=(1, 2)) > 1e-3)   # 7, 8, 9


def test_bad_chunks_are_rejected():
    with pytest.raises(ValueError):
        opf.query_positions([0, 5], [4])                # chunk longer than the context
    with pytest.raises(ValueError):
        opf.query_positions([1, 5], [9])


def test_prefill_workload_replay_equals_contiguous_causal():
    """The prefill workload's replay (cached prefix, then each entry's chunk
    appended in order) gives each chunk query causal attention over its own
    request's tokens, here checked against SDPA on the request's history."""
    torch = pytest.importorskip("torch")
    from oracle import replay as orp
    from paged_kv_cache_253_gb300 import workloads as wls
    wl = wls.make_workload("prefill", num_seqs=3, lengths=[0, 5, 17], chunks=[6, 1, 9],
                           num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4)
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    assert st.cu_seqlens_q.tolist() == [0, 6, 7, 16]
    assert st.context_lens.tolist() == [6, 6, 26]
    out = orp.prefill_attention(wl, values, st)
    hk = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["hist_k"]))
    hv = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["hist_v"]))
    nk = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["new_k"]))
    nv = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["new_v"]))
    q = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["q"]))
    hist = [0, 0, 5]
    for s, (P, n) in enumerate(zip([0, 5, 17], [6, 1, 9])):
        ks = np.concatenate([hk[hist[s]:hist[s] + P], nk[st.cu_seqlens_q[s]:st.cu_seqlens_q[s + 1]]])
        vs = np.concatenate([hv[hist[s]:hist[s] + P], nv[st.cu_seqlens_q[s]:st.cu_seqlens_q[s + 1]]])
        qs = q[st.cu_seqlens_q[s]:st.cu_seqlens_q[s + 1]]
        # causal attention of the chunk rows, as the last n rows of a full square mask
        L = P + n
        mask = np.tril(np.ones((L, L), dtype=bool))[P:]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qs.astype(np.float64)).permute(1, 0, 2),
            torch.from_numpy(ks.astype(np.float64)).permute(1, 0, 2).repeat_interleave(2, 0),
            torch.from_numpy(vs.astype(np.float64)).permute(1, 0, 2).repeat_interleave(2, 0),
            attn_mask=torch.from_numpy(mask), scale=wl.scale)
        np.testing.assert_allclose(out[st.cu_seqlens_q[s]:st.cu_seqlens_q[s + 1]],
                                   ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_prefill_after_a_fork_copies_the_shared_partial_block():
    """Two requests share a 10-token prompt (block size 4: the third block is
    partly filled and shared); each then prefills its own chunk.  The first
    chunk token of the first request copies the shared partial block (the
    second request, the last holder, writes in place), and each request's
    queries see only its own chunk on top of the shared prompt."""
    torch = pytest.importorskip("torch")
    from oracle import replay as orp
    from paged_kv_cache_253_gb300 import workloads as wls
    rng = np.random.default_rng(12)
    prompt = rng.integers(0, 100, size=10).astype(np.int32)
    chunks = np.array([5, 3], np.int32)
    wl = wls.Workload(name="prefill", block_size=4, num_q_heads=4, num_kv_heads=2, head_dim=8,
                      dtype="bf16", num_blocks=12,
                      free_order=rng.permutation(12).astype(np.int32),
                      events=[("add", 0, prompt, 0), ("extend", 0, prompt), ("fork", 1, 0)],
                      batch=np.array([0, 1], np.int32),
                      step_tokens=rng.integers(0, 100, size=8).astype(np.int32),
                      scale=0.35, seed=12, chunk_lens=chunks)
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    assert len(st.step_pairs) == 1                       # one copy-on-write, by request 0
    t0, t1 = st.block_tables
    assert t0[0] == t1[0] and t0[1] == t1[1] and t0[2] != t1[2]
    assert st.context_lens.tolist() == [15, 13]
    out = orp.prefill_attention(wl, values, st)
    hk = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["hist_k"]))
    hv = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["hist_v"]))
    nk = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["new_k"]))
    nv = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["new_v"]))
    q = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["q"]))
    cu = [0, 5, 8]
    for s in range(2):
        ks = np.concatenate([hk, nk[cu[s]:cu[s + 1]]]).astype(np.float64)
        vs = np.concatenate([hv, nv[cu[s]:cu[s + 1]]]).astype(np.float64)
        L, n = 10 + chunks[s], chunks[s]
        mask = np.tril(np.ones((L, L), dtype=bool))[L - n:]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[cu[s]:cu[s + 1]].astype(np.float64)).permute(1, 0, 2),
            torch.from_numpy(ks).permute(1, 0, 2).repeat_interleave(2, 0),
            torch.from_numpy(vs).permute(1, 0, 2).repeat_interleave(2, 0),
            attn_mask=torch.from_numpy(mask), scale=0.35)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_fp8_prefill_replay_equals_contiguous_causal_over_quantized_rows():
    """An fp8 pool stores every appended row (history and chunk) as codes under
    its own K or V scale; the prefill oracle reads the values the codes stand
    for: each chunk query equals causal attention over its request's rows,
    each quantized on its own (K and V scales differ, so a swap shows)."""
    torch = pytest.importorskip("torch")
    from oracle import fp8
    from oracle import replay as orp
    from paged_kv_cache_253_gb300 import workloads as wls
    wl = wls.make_workload("prefill", num_seqs=3, lengths=[0, 5, 17], chunks=[6, 1, 9],
                           num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4, dtype="fp8")
    assert wl.kv_scales[0] != wl.kv_scales[1]
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    assert st.k_pool.dtype == np.uint8
    out = orp.prefill_attention(wl, values, st)

    def rows(name, which):
        x = oatt.bf16_bits_to_f32(orp.values_to_numpy(values[name]))
        return fp8.dequantize(fp8.quantize(x, wl.kv_scales[which]), wl.kv_scales[which])
    hk, hv, nk, nv = rows("hist_k", 0), rows("hist_v", 1), rows("new_k", 0), rows("new_v", 1)
    q = oatt.bf16_bits_to_f32(orp.values_to_numpy(values["q"]))
    hist = [0, 0, 5]
    for s, (P, n) in enumerate(zip([0, 5, 17], [6, 1, 9])):
        c0, c1 = st.cu_seqlens_q[s], st.cu_seqlens_q[s + 1]
        ks = np.concatenate([hk[hist[s]:hist[s] + P], nk[c0:c1]])
        vs = np.concatenate([hv[hist[s]:hist[s] + P], nv[c0:c1]])
        L = P + n
        mask = np.tril(np.ones((L, L), dtype=bool))[P:]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[c0:c1].astype(np.float64)).permute(1, 0, 2),
            torch.from_numpy(ks.astype(np.float64)).permute(1, 0, 2).repeat_interleave(2, 0),
            torch.from_numpy(vs.astype(np.float64)).permute(1, 0, 2).repeat_interleave(2, 0),
            attn_mask=torch.from_numpy(mask), scale=wl.scale)
        np.testing.assert_allclose(out[c0:c1], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
    # the bf16 workload's prefill differs from it by quantization error only
    # (e4m3 keeps 3 mantissa bits: a few-key row can move by several percent
    # of a value)
    wl16 = wls.make_workload("prefill", num_seqs=3, lengths=[0, 5, 17], chunks=[6, 1, 9],
                             num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4)
    ref16 = orp.prefill_attention(wl16, values, orp.replay(wl16, values))
    err = np.abs(out - ref16).max()
    assert 1e-4 < err < 0.5, err
