"""GPU parity: the library (C++ block manager + CUDA kernels, called through the
C ABI) against the oracle (naive bookkeeping + float64 loops), on the same
seeded inputs.

* bookkeeping (slots, copy pairs, block tables, lengths) — bit-exact;
* pool contents after every copy-on-write copy and append — bit-exact;
* attention output — max-abs error <= 1e-5 (fp32 pool) or <= 5e-3 (bf16).
"""
import numpy as np
import pytest
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import workloads as wls

from gpu_common import assert_pools_equal, run_library, tol

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)

SMALL = [
    ("tiny", dict()),
    ("decode", dict(num_seqs=6, min_len=1, max_len=300, **D128)),
    ("decode", dict(num_seqs=5, min_len=1, max_len=200, num_q_heads=64, num_kv_heads=8,
                    head_dim=128)),                                     # G = 8
    ("decode", dict(num_seqs=4, min_len=1, max_len=150, num_q_heads=8, num_kv_heads=8,
                    head_dim=128)),                                     # G = 1
    ("decode", dict(num_seqs=4, min_len=1, max_len=150, num_q_heads=10, num_kv_heads=2,
                    head_dim=128)),                                     # G = 5
    ("decode", dict(num_seqs=4, min_len=1, max_len=200, num_q_heads=16, num_kv_heads=4,
                    head_dim=64)),
    ("decode", dict(num_seqs=3, min_len=1, max_len=200, num_q_heads=8, num_kv_heads=2,
                    head_dim=256)),
    ("decode", dict(num_seqs=4, min_len=1, max_len=200, block_size=32, **D128)),
    ("decode", dict(num_seqs=4, min_len=1, max_len=100, block_size=8, **D128)),   # fp32 path
    ("decode", dict(num_seqs=4, min_len=1, max_len=100, dtype="f32", **D128)),
    ("decode", dict(num_seqs=3, min_len=1, max_len=100, num_q_heads=32, num_kv_heads=2,
                    head_dim=128)),                                     # G = 16
    ("decode", dict(lengths=[0, 1, 15, 16, 17, 33], **D128)),
    ("prefix", dict(num_seqs=6, prefix_len=41, suffix_min=1, suffix_max=40, **D128)),
    ("mixed", dict(num_seqs=24, median=60, min_len=1, max_len=400, prefix_min=20,
                   prefix_max=90, num_q_heads=64, num_kv_heads=8, head_dim=128)),
    ("long", dict(num_seqs=2, min_len=3000, max_len=9000, **D128)),
]


def _ids():
    out = []
    for name, kw in SMALL:
        tag = "-".join(f"{k}{v}" for k, v in kw.items() if k not in ("num_q_heads",))
        out.append(f"{name}-{tag}"[:60])
    return out


def _check(wl, values, seqs=None, threads=1, shared=True):
    pool, bm, setup_pairs, step = run_library(wl, values, shared=shared)
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    # bookkeeping, bit-exact
    assert setup_pairs == st.setup_pairs
    assert step.slots.cpu().numpy().tolist() == st.step_slots.tolist()
    assert [tuple(p) for p in step.pairs.cpu().numpy().tolist()] == st.step_pairs
    assert np.array_equal(step.block_tables.cpu().numpy(), st.block_tables)
    assert np.array_equal(step.context_lens.cpu().numpy(), st.context_lens)
    # pool contents, bit-exact
    assert_pools_equal(pool, st)
    # attention
    ref = orp.attention(wl, values, st, seqs=seqs, threads=threads)
    got = step.out.double().cpu().numpy()
    if seqs is not None:
        got = got[np.asarray(seqs)]
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"
    return err, pool, step


@pytest.mark.parametrize("name,kw", SMALL, ids=_ids())
def test_small_parity(name, kw):
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cpu")
    err, pool, step = _check(wl, values)
    print(f"{name} {kw}: max-abs {err:.3g}")


def test_repeated_step_is_idempotent():
    wl = wls.make_workload("prefix", num_seqs=5, prefix_len=37, suffix_min=0, suffix_max=0,
                           **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    first = step.out.clone()
    assert step.num_pairs == 4          # every fork but the last copies the partial block
    for _ in range(3):
        step.run()
    torch.cuda.synchronize()
    assert torch.equal(first, step.out)
    assert pool.get_error() == 0


def test_moving_physical_blocks_leaves_output_unchanged():
    wl = wls.make_workload("decode", num_seqs=6, min_len=1, max_len=400, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    base = step.out.clone()
    k, v = pool.export()
    move = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(5)).cuda()
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    k2[move] = k
    v2[move] = v
    pool.import_(k2, v2)
    t = step.block_tables
    t2 = torch.where(t >= 0, move[t.clamp(min=0).long()].int(), t).contiguous()
    out = pool.decode(step.q, t2, step.context_lens, step.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, base)
    assert pool.get_error() == 0


def test_sorted_tables_change_the_output():
    wl = wls.make_workload("decode", lengths=[40, 70], **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    t = step.block_tables.clone()
    n = (t >= 0).sum(1)
    for i in range(t.shape[0]):
        t[i, :n[i]] = t[i, :n[i]].sort(descending=True).values
    out = pool.decode(step.q, t.contiguous(), step.context_lens, step.scale)
    torch.cuda.synchronize()
    assert (out - step.out).abs().max().item() > 1e-3


def test_bf16_output_dtype():
    wl = wls.make_workload("decode", num_seqs=4, min_len=1, max_len=300, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    out16 = pool.decode(step.q, step.block_tables, step.context_lens, step.scale,
                        out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out16, step.out.to(torch.bfloat16))


def test_device_errors_are_reported_not_faulted():
    from paged_kv_cache_253_gb300._lib import (PA_ERR_BAD_BLOCK_ID, PA_ERR_BAD_LENGTH,
                                               PA_ERR_BAD_SLOT, PA_ERR_OVERLAP)
    wl = wls.make_workload("decode", num_seqs=3, min_len=20, max_len=60, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    assert pool.get_error() == 0
    bad = step.block_tables.clone()
    bad[1, 0] = wl.num_blocks + 5
    pool.decode(step.q, bad, step.context_lens, step.scale)
    assert pool.get_error() == PA_ERR_BAD_BLOCK_ID
    assert pool.get_error() == 0                       # cleared by the read
    long_lens = step.context_lens.clone()
    long_lens[0] = bad.shape[1] * wl.block_size + 100
    pool.decode(step.q, step.block_tables, long_lens, step.scale)
    assert pool.get_error() == PA_ERR_BAD_LENGTH
    slots = torch.tensor([wl.num_blocks * wl.block_size + 3, -1, 0], dtype=torch.int64,
                         device="cuda")
    pool.append_kv(step.new_k, step.new_v, slots)
    assert pool.get_error() == PA_ERR_BAD_SLOT
    pairs = torch.tensor([[1, 2], [2, 3]], dtype=torch.int64, device="cuda")
    pool.copy_blocks(pairs)
    assert pool.get_error() == PA_ERR_OVERLAP
    pairs = torch.tensor([[1, wl.num_blocks]], dtype=torch.int64, device="cuda")
    pool.copy_blocks(pairs)
    assert pool.get_error() == PA_ERR_BAD_BLOCK_ID


def test_copy_blocks_skips_only_conflicting_pairs():
    wl = wls.make_workload("decode", num_seqs=2, min_len=40, max_len=60, pool_factor=4.0,
                           **D128)
    assert wl.num_blocks >= 12
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    k0, v0 = pool.export()
    pairs = torch.tensor([[0, 5], [7, 9], [9, 11]], dtype=torch.int64, device="cuda")
    pool.copy_blocks(pairs)
    torch.cuda.synchronize()
    k1, v1 = pool.export()
    torch.cuda.synchronize()
    assert torch.equal(k1[5], k0[0]) and torch.equal(v1[5], v0[0])
    assert torch.equal(k1[9], k0[9]) and torch.equal(k1[11], k0[11])   # conflicting: untouched
    assert pool.get_error() != 0


@pytest.mark.parametrize("name,kw", [SMALL[1], SMALL[5], SMALL[8], SMALL[11], SMALL[12],
                                     SMALL[13]], ids=lambda x: str(x)[:40])
def test_fused_append_matches_separate_calls(name, kw):
    """pa_append_decode leaves the same pool bits and output as pa_append_kv
    followed by pa_decode."""
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cpu")
    outs, pools = [], []
    for fused in (False, True):
        pool, bm, _, step = run_library(wl, values, shared=False, fused=fused)
        assert pool.get_error() == 0
        outs.append(step.out.clone())
        pools.append(pool.export())
    torch.cuda.synchronize()
    assert torch.equal(pools[0][0], pools[1][0]) and torch.equal(pools[0][1], pools[1][1])
    assert torch.equal(outs[0], outs[1])


def test_fused_append_rejects_a_foreign_slot():
    from paged_kv_cache_253_gb300._lib import PA_ERR_INVALID_ARG
    wl = wls.make_workload("decode", num_seqs=3, min_len=20, max_len=60, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    assert pool.get_error() == 0
    wrong = step.slots.clone()
    wrong[0], wrong[1] = step.slots[1], step.slots[0]
    pool.append_decode(step.new_k, step.new_v, wrong, step.q, step.block_tables,
                       step.context_lens, step.scale)
    assert pool.get_error() == PA_ERR_INVALID_ARG


# ------------------------------------------------------- shared prefix ---

SHARED_CASES = [
    ("prefix", dict(num_seqs=6, prefix_len=300, suffix_min=1, suffix_max=40, **D128)),
    ("prefix", dict(num_seqs=70, prefix_len=1030, suffix_min=0, suffix_max=30, **D128)),
    ("prefix", dict(num_seqs=9, prefix_len=700, suffix_min=5, suffix_max=60, num_q_heads=64,
                    num_kv_heads=8, head_dim=128)),                              # G = 8
    ("prefix", dict(num_seqs=5, prefix_len=500, suffix_min=1, suffix_max=9, num_q_heads=10,
                    num_kv_heads=2, head_dim=128)),                              # G = 5
    ("prefix", dict(num_seqs=5, prefix_len=640, suffix_min=1, suffix_max=70, block_size=32,
                    num_q_heads=16, num_kv_heads=4, head_dim=64)),
    ("mixed", dict(num_seqs=40, median=60, min_len=1, max_len=600, prefix_min=100,
                   prefix_max=900, num_q_heads=64, num_kv_heads=8, head_dim=128)),
]


@pytest.mark.parametrize("name,kw", SHARED_CASES, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SHARED_CASES)])
def test_shared_prefix_parity(name, kw):
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cpu")
    err, pool, step = _check(wl, values, shared=True)
    offs, seqs, nsh = step.groups
    assert len(nsh) >= 1 and nsh.min() >= 1, "the workload must have a shared span"
    plain = pool.decode(step.q, step.block_tables, step.context_lens, step.scale)
    torch.cuda.synchronize()
    diff = (plain - step.out).abs().max().item()
    assert diff <= 1e-4, f"shared vs plain decode differ by {diff:.3g}"
    print(f"{name} {kw}: groups {len(nsh)} shared blocks {nsh.tolist()} max-abs {err:.3g}")


def test_shared_description_is_checked_on_the_device():
    from paged_kv_cache_253_gb300._lib import PA_ERR_INVALID_ARG
    wl = wls.make_workload("prefix", num_seqs=4, prefix_len=100, suffix_min=1, suffix_max=5,
                           **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values)
    assert pool.get_error() == 0
    offs, seqs, nsh = step.groups
    bad_tables = step.block_tables.clone()
    bad_tables[int(seqs[1]), 0] = bad_tables[int(seqs[1]), 1]      # members disagree
    pool.decode_shared(step.q, bad_tables.contiguous(), step.context_lens, step.scale,
                       (offs, seqs, nsh))
    assert pool.get_error() == PA_ERR_INVALID_ARG
    from paged_kv_cache_253_gb300._lib import PagedAttnError
    with pytest.raises(PagedAttnError):                                # beyond the table: host
        pool.decode_shared(step.q, step.block_tables, step.context_lens, step.scale,
                           (offs, seqs, nsh + 50))
    assert nsh[0] + 1 <= step.block_tables.shape[1]
    pool.decode_shared(step.q, step.block_tables, step.context_lens, step.scale,
                       (offs, seqs, nsh + 1))                          # beyond the contexts: device
    assert pool.get_error() == PA_ERR_INVALID_ARG
    out = pool.decode_shared(step.q, step.block_tables, step.context_lens, step.scale,
                             (offs, seqs, nsh))
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    assert torch.allclose(out, step.out, atol=1e-6, rtol=0)


# ---------------------------------------------------------- full sizes ---

def _sample(wl, n=10):
    """Batch entries whose outputs the oracle recomputes: longest, shortest,
    shared ones, and a seeded spread."""
    rng = np.random.default_rng(wl.seed)
    S = wl.num_seqs
    pick = set(rng.choice(S, size=min(n, S), replace=False).tolist())
    pick |= {0, S - 1}
    return sorted(pick)


FULL_CASES = [("decode", False), ("long", False), ("prefix", False), ("prefix", True),
              ("mixed", False), ("mixed", True)]


@pytest.mark.parametrize("name,shared", FULL_CASES, ids=[f"{n}-{'shared' if s else 'plain'}"
                                                          for n, s in FULL_CASES])
def test_full_size_parity(name, shared):
    wl = wls.make_workload(name)
    values = wls.generate_values(wl, "cuda")
    seqs = _sample(wl)
    if name == "long":
        seqs = list(range(wl.num_seqs))
    err, pool, step = _check(wl, values, seqs=seqs, threads=8, shared=shared)
    print(f"{name} shared={shared}: max-abs over {len(seqs)} sampled sequences {err:.3g}")
