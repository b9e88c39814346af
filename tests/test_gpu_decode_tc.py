"""The tcgen05 decode split kernel (pool option decode_kernel = 2) against the
oracle (GPU).

The kernel computes what the mma.sync split kernels compute (kgptalkie "Day
28: PagedAttention / vLLM", "Follow One Token Address": every query scores the
keys its request's table and length name, in logical order) with the cached
tokens as the tensor-core product's M dimension.  These tests run it on bf16
and fp8 pools: outputs against the float64 oracle, pools bit-exact after
pa_append_decode (the append happens inside the kernel), a foreign slot
refused, blocks with bad ids reported, stale NaN/Inf never reaching an output,
and a captured step replaying bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import runtime, workloads as wls

from gpu_common import assert_pools_equal, tol

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)
TC = 2          # decode_kernel option value: tcgen05 where the shape allows it


def _run(wl, values, opt=TC, fused=True):
    pool, bm, setup_pairs = runtime.replay_setup(wl, values, "cuda")
    pool.set_option("decode_kernel", opt)
    step = runtime.prepare_step(wl, values, pool, bm, shared=False, fused=fused)
    step.run()
    torch.cuda.synchronize()
    return pool, step


CASES = [
    ("decode", dict(lengths=[0, 1, 15, 16, 17, 33, 127, 128, 129, 300], **D128)),
    ("decode", dict(num_seqs=6, min_len=1, max_len=3000, **D128)),
    ("decode", dict(num_seqs=5, min_len=1, max_len=700, num_q_heads=64, num_kv_heads=8,
                    head_dim=128)),                                      # G = 8
    ("decode", dict(num_seqs=4, min_len=1, max_len=500, num_q_heads=8, num_kv_heads=8,
                    head_dim=128)),                                      # G = 1
    ("decode", dict(num_seqs=4, min_len=1, max_len=500, num_q_heads=10, num_kv_heads=2,
                    head_dim=128)),                                      # G = 5
    ("long", dict(num_seqs=2, min_len=3000, max_len=9000, **D128)),
    ("mixed", dict(num_seqs=24, median=60, min_len=1, max_len=400, prefix_min=20,
                   prefix_max=90, num_q_heads=64, num_kv_heads=8, head_dim=128)),
]
FP8 = [(n, dict(kw, dtype="fp8")) for n, kw in CASES if n != "mixed"]


@pytest.mark.parametrize("name,kw", CASES + FP8,
                         ids=[f"{n}{i}-{kw.get('dtype', 'bf16')}" for i, (n, kw) in enumerate(CASES + FP8)])
def test_tc_decode_parity(name, kw):
    """Output against the oracle, and the pool bit-exact after the fused append."""
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cpu")
    pool, step = _run(wl, values)
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert_pools_equal(pool, st)
    ref = orp.attention(wl, values, st, threads=8)
    got = step.out.double().cpu().numpy()
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_tc_matches_mma_sync(dtype):
    """Both split kernels, same step: the same pools bit for bit, outputs
    within the tolerance of each other."""
    wl = wls.make_workload("decode", num_seqs=12, min_len=1, max_len=2500, dtype=dtype, **D128)
    values = wls.generate_values(wl, "cpu")
    outs, pools = [], []
    for opt in (1, TC):
        pool, step = _run(wl, values, opt=opt)
        assert pool.get_error() == 0
        outs.append(step.out.double().cpu().numpy())
        pools.append(pool.export())
    torch.cuda.synchronize()
    assert torch.equal(pools[0][0], pools[1][0]) and torch.equal(pools[0][1], pools[1][1])
    assert np.abs(outs[0] - outs[1]).max() <= tol(wl)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_tc_fused_append_equals_separate_calls(dtype):
    wl = wls.make_workload("decode", num_seqs=7, min_len=1, max_len=900, dtype=dtype, **D128)
    values = wls.generate_values(wl, "cpu")
    res = []
    for fused in (False, True):
        pool, step = _run(wl, values, fused=fused)
        assert pool.get_error() == 0
        res.append((step.out.clone(), pool.export()))
    torch.cuda.synchronize()
    (o0, (k0, v0)), (o1, (k1, v1)) = res
    assert torch.equal(k0, k1) and torch.equal(v0, v1)
    assert torch.equal(o0, o1)


def test_tc_fused_append_rejects_a_foreign_slot():
    from paged_kv_cache_253_gb300._lib import PA_ERR_INVALID_ARG
    wl = wls.make_workload("decode", num_seqs=3, min_len=20, max_len=60, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, step = _run(wl, values)
    assert pool.get_error() == 0
    wrong = step.slots.clone()
    wrong[0], wrong[1] = step.slots[1], step.slots[0]
    pool.append_decode(step.new_k, step.new_v, wrong, step.q, step.block_tables,
                       step.context_lens, step.scale)
    assert pool.get_error() == PA_ERR_INVALID_ARG


def test_tc_bad_block_id_is_reported_not_faulted():
    from paged_kv_cache_253_gb300._lib import PA_ERR_BAD_BLOCK_ID
    wl = wls.make_workload("decode", num_seqs=4, min_len=40, max_len=400, **D128)
    values = wls.generate_values(wl, "cpu")
    pool, step = _run(wl, values)
    assert pool.get_error() == 0
    tables = step.block_tables.clone()
    tables[1, 1] = pool.num_blocks + 5
    tables[2, 0] = -3
    pool.decode(step.q, tables, step.context_lens, step.scale, out=step.out)
    assert pool.get_error() == PA_ERR_BAD_BLOCK_ID


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_tc_ignores_stale_nonfinite(dtype):
    from test_gpu_nonfinite import _plant
    wl = wls.make_workload("decode", lengths=[1, 15, 17, 33, 100, 250, 129], dtype=dtype, **D128)
    values = wls.generate_values(wl, "cuda")
    pool, step = _run(wl, values)
    assert pool.get_error() == 0
    assert _plant(pool, step.block_tables.cpu().numpy(), step.context_lens.cpu().numpy()) > 0
    step.out.fill_(float("nan"))
    step.decode()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    got = step.out.double().cpu().numpy()
    assert np.isfinite(got).all(), "a planted non-finite value reached the output"
    st = orp.replay(wl, values)
    ref = orp.attention(wl, values, st, threads=4)
    assert np.abs(got - ref).max() <= tol(wl)


def test_tc_graph_replay_is_bit_exact():
    wl = wls.make_workload("decode", num_seqs=9, min_len=1, max_len=1500, **D128)
    values = wls.generate_values(wl, "cuda")
    pool, step = _run(wl, values)
    ref = step.out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    step.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    assert torch.equal(step.out, ref)


@pytest.mark.parametrize("name,dtype", [("decode", "bf16"), ("decode", "fp8"), ("long", "bf16"),
                                        ("long", "fp8"), ("mixed", "bf16")])
def test_tc_full_size_parity(name, dtype):
    """The bench's workloads at full size, sampled sequences against the oracle."""
    wl = wls.make_workload(name, dtype=dtype)
    values = wls.generate_values(wl, "cpu")
    pool, step = _run(wl, values)
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    seqs = sorted(set(np.random.default_rng(7).integers(0, wl.num_seqs, 4).tolist() + [wl.num_seqs - 1]))
    ref = orp.attention(wl, values, st, seqs=seqs, threads=16)
    got = step.out.double().cpu().numpy()[seqs]
    err = np.abs(got - ref).max()
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"
