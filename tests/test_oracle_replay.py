"""The oracle's replay of whole workloads equals contiguous attention over each
request's own token history (kgptalkie "Day 28", verification recipe under "A
Tiny Block-Table Example"), including requests that share blocks and diverge by
copy-on-write.  CPU only."""
import numpy as np
import pytest

from oracle import attention as oa
from oracle import fp8
from oracle import replay as orp
from paged_kv_cache_253_gb300 import workloads as wls


def _histories(wl, values):
    """Each batch request's keys/values in token order, from the script alone."""
    hk = orp.values_to_numpy(values["hist_k"])
    hv = orp.values_to_numpy(values["hist_v"])
    nk = orp.values_to_numpy(values["new_k"])
    nv = orp.values_to_numpy(values["new_v"])
    rows = {}
    r = 0
    for ev in wl.events:
        if ev[0] == "add":
            rows[ev[1]] = []
        elif ev[0] == "fork":
            rows[ev[1]] = list(rows[ev[2]])
        elif ev[0] == "extend":
            n = len(ev[2])
            rows[ev[1]].extend(range(r, r + n))
            r += n
    ks, vs = [], []
    for i, rid in enumerate(wl.batch.tolist()):
        idx = np.asarray(rows[rid], dtype=np.int64)
        ks.append(np.concatenate([hk[idx], nk[i:i + 1]]))
        vs.append(np.concatenate([hv[idx], nv[i:i + 1]]))
    return ks, vs


CASES = [
    ("tiny", {}),
    ("decode", dict(num_seqs=5, min_len=1, max_len=70, num_q_heads=8, num_kv_heads=2,
                    head_dim=16)),
    ("prefix", dict(num_seqs=6, prefix_len=41, suffix_min=1, suffix_max=20, num_q_heads=4,
                    num_kv_heads=2, head_dim=16)),
    ("mixed", dict(num_seqs=20, median=30, min_len=1, max_len=90, prefix_min=20,
                   prefix_max=50, num_q_heads=8, num_kv_heads=2, head_dim=16)),
    ("long", dict(num_seqs=2, min_len=200, max_len=300, num_q_heads=4, num_kv_heads=1,
                  head_dim=16)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_replay_equals_contiguous(name, kw):
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    paged = orp.attention(wl, values, st)
    ks, vs = _histories(wl, values)
    q = orp.values_to_numpy(values["q"])
    if q.dtype == np.uint16:
        q = oa.bf16_bits_to_f32(q)
    contig = oa.contiguous_decode(q, ks, vs, wl.scale, wl.num_kv_heads)
    np.testing.assert_array_equal(paged, contig)
    assert st.context_lens.tolist() == [k.shape[0] for k in ks]


FP8_CASES = [
    ("decode", dict(num_seqs=5, min_len=1, max_len=70, num_q_heads=8, num_kv_heads=2,
                    head_dim=16, dtype="fp8")),
    ("mixed", dict(num_seqs=20, median=30, min_len=1, max_len=90, prefix_min=20,
                   prefix_max=50, num_q_heads=8, num_kv_heads=2, head_dim=16, dtype="fp8")),
]


@pytest.mark.parametrize("name,kw", FP8_CASES, ids=[c[0] for c in FP8_CASES])
def test_fp8_replay_equals_contiguous_over_quantized_rows(name, kw):
    """An fp8 pool holds each appended row's codes under its own scale (K and V
    differ), and the paged attention reads their values: equal to contiguous
    attention over the same rows quantized one by one, here."""
    wl = wls.make_workload(name, **kw)
    assert wl.kv_scales[0] != wl.kv_scales[1]
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    assert st.k_pool.dtype == np.uint8
    paged = orp.attention(wl, values, st)
    ks, vs = _histories(wl, values)
    ks = [fp8.dequantize(fp8.quantize(oa.bf16_bits_to_f32(k), wl.kv_scales[0]), wl.kv_scales[0])
          for k in ks]
    vs = [fp8.dequantize(fp8.quantize(oa.bf16_bits_to_f32(v), wl.kv_scales[1]), wl.kv_scales[1])
          for v in vs]
    q = oa.bf16_bits_to_f32(orp.values_to_numpy(values["q"]))
    contig = oa.contiguous_decode(q, ks, vs, wl.scale, wl.num_kv_heads)
    np.testing.assert_array_equal(paged, contig)
    # the same step over the unquantized bf16 rows differs by quantization error only
    wl16 = wls.make_workload(name, **{**kw, "dtype": "bf16"})
    ref16 = orp.attention(wl16, values, orp.replay(wl16, values))
    err = np.abs(paged - ref16).max()
    assert 1e-4 < err < 0.1, err


def test_tiny_workload_shape():
    wl = wls.make_workload("tiny")
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    assert st.context_lens.tolist() == [10, 4, 6]
    assert [int((t >= 0).sum()) for t in st.block_tables] == [3, 1, 2]
    used = st.block_tables[st.block_tables >= 0]
    assert len(set(used.tolist())) == used.size and used.max() < 16


def test_prefix_divergence_pairs():
    wl = wls.make_workload("prefix", num_seqs=8, prefix_len=4104, suffix_min=1, suffix_max=3,
                           num_q_heads=2, num_kv_heads=1, head_dim=8)
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    assert len(st.setup_pairs) == 7 and st.step_pairs == []
    full = st.block_tables[:, :256]
    assert (full == full[0]).all()
    assert all(st.bm.refcount[b] == 8 for b in full[0])


def test_mixed_step_copies_for_mid_block_divergence():
    wl = wls.make_workload("mixed", num_seqs=40, median=30, min_len=1, max_len=90,
                           prefix_min=20, prefix_max=50, num_q_heads=4, num_kv_heads=1,
                           head_dim=8)
    values = wls.generate_values(wl, "cpu")
    st = orp.replay(wl, values)
    expect = 0
    for grp in wl.shared_groups:
        root_len = [len(e[2]) for e in wl.events if e[0] == "extend" and e[1] == grp[0]][0]
        if root_len % wl.block_size:
            expect += len(grp) - 1
    assert len(st.step_pairs) == expect and expect > 0
