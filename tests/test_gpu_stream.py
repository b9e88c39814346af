"""GPU parity of the stream-K decode split pass (PA_DECODE_STREAM=1): equal
tile ranges per warp, TMA-fed per-warp rings, pieces merged by the last warp
to finish one.  Same oracle and tolerances as the default path; the library
reads the switch on every decode call."""
import numpy as np
import pytest
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import workloads as wls

from gpu_common import assert_pools_equal, run_library, tol

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)

CASES = [
    ("decode", dict(num_seqs=6, min_len=1, max_len=300, **D128)),
    ("decode", dict(num_seqs=5, min_len=1, max_len=200, num_q_heads=64, num_kv_heads=8,
                    head_dim=128)),                                     # G = 8
    ("decode", dict(num_seqs=4, min_len=1, max_len=150, num_q_heads=8, num_kv_heads=8,
                    head_dim=128)),                                     # G = 1
    ("decode", dict(num_seqs=4, min_len=1, max_len=150, num_q_heads=10, num_kv_heads=2,
                    head_dim=128)),                                     # G = 5
    ("decode", dict(num_seqs=4, min_len=1, max_len=200, num_q_heads=16, num_kv_heads=4,
                    head_dim=64)),
    ("decode", dict(lengths=[0, 1, 15, 16, 17, 33], **D128)),           # empty and ragged
    ("decode", dict(num_seqs=40, min_len=1, max_len=2500, **D128)),     # pieces over many warps
    ("long", dict(num_seqs=2, min_len=3000, max_len=9000, **D128)),
    ("mixed", dict(num_seqs=24, median=60, min_len=1, max_len=400, prefix_min=20,
                   prefix_max=90, num_q_heads=64, num_kv_heads=8, head_dim=128)),
]


@pytest.fixture
def stream(monkeypatch):
    monkeypatch.setenv("PA_DECODE_STREAM", "1")


def _check(wl, values, seqs=None, threads=1, fused=True):
    pool, bm, setup_pairs, step = run_library(wl, values, shared=False, fused=fused)
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert step.slots.cpu().numpy().tolist() == st.step_slots.tolist()
    assert_pools_equal(pool, st)
    ref = orp.attention(wl, values, st, seqs=seqs, threads=threads)
    got = step.out.double().cpu().numpy()
    if seqs is not None:
        got = got[np.asarray(seqs)]
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"
    return err, pool, step


@pytest.mark.parametrize("name,kw", CASES, ids=[f"{n}-{i}" for i, (n, _) in enumerate(CASES)])
def test_stream_parity(stream, name, kw):
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cpu")
    err, pool, step = _check(wl, values)
    print(f"stream {name}: max-abs {err:.3g}")


@pytest.mark.parametrize("name,kw", [CASES[0], CASES[5], CASES[6], CASES[8]],
                         ids=["decode", "ragged", "many-warps", "mixed"])
def test_stream_fused_append_matches_separate_calls(stream, name, kw):
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


def test_stream_repeated_steps_reset_their_counters(stream):
    """The unit arrival counters reset themselves: the same step run again gives
    the same bits."""
    wl = wls.make_workload("decode", num_seqs=40, min_len=1, max_len=2500, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values, shared=False, fused=False)
    first = step.decode().clone()
    for _ in range(4):
        again = step.decode()
        torch.cuda.synchronize()
        assert torch.equal(again, first)
    assert pool.get_error() == 0


def test_stream_matches_default_path(monkeypatch):
    wl = wls.make_workload("decode", num_seqs=30, min_len=1, max_len=1500, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values, shared=False, fused=False)
    monkeypatch.setenv("PA_DECODE_STREAM", "0")
    base = step.decode().clone()
    monkeypatch.setenv("PA_DECODE_STREAM", "1")
    got = step.decode().clone()
    torch.cuda.synchronize()
    assert (got - base).abs().max().item() <= 1e-5
    assert pool.get_error() == 0


def test_stream_device_errors(stream):
    from paged_kv_cache_253_gb300._lib import (PA_ERR_BAD_BLOCK_ID, PA_ERR_BAD_LENGTH,
                                               PA_ERR_INVALID_ARG)
    wl = wls.make_workload("decode", num_seqs=3, min_len=20, max_len=60, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _, step = run_library(wl, values, shared=False)
    assert pool.get_error() == 0
    bad = step.block_tables.clone()
    bad[1, 0] = wl.num_blocks + 5
    pool.decode(step.q, bad, step.context_lens, step.scale)
    assert pool.get_error() == PA_ERR_BAD_BLOCK_ID
    long_lens = step.context_lens.clone()
    long_lens[0] = bad.shape[1] * wl.block_size + 100
    pool.decode(step.q, step.block_tables, long_lens, step.scale)
    assert pool.get_error() == PA_ERR_BAD_LENGTH
    wrong = step.slots.clone()
    wrong[0], wrong[1] = step.slots[1], step.slots[0]
    pool.append_decode(step.new_k, step.new_v, wrong, step.q, step.block_tables,
                       step.context_lens, step.scale)
    assert pool.get_error() == PA_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["decode", "long", "mixed"])
def test_stream_full_size_parity(stream, name):
    wl = wls.make_workload(name)
    values = wls.generate_values(wl, "cuda")
    rng = np.random.default_rng(wl.seed)
    S = wl.num_seqs
    seqs = sorted(set(rng.choice(S, size=min(10, S), replace=False).tolist()) | {0, S - 1})
    if name == "long":
        seqs = list(range(S))
    err, pool, step = _check(wl, values, seqs=seqs, threads=8)
    print(f"stream {name}: max-abs over {len(seqs)} sampled sequences {err:.3g}")
