"""Stale non-finite bits outside every context never reach an output (GPU).

A physical block recycled from a finished request keeps whatever that request
wrote: the positions past its new owner's context length, and whole blocks on
the free list, may hold Inf or NaN.  The attention kernels read whole 16-token
tiles and weigh the positions past a context by zero, and 0 * Inf is NaN, so
each kernel must keep those bits out of its value product (masking the value
fragments, or zeroing the staged value columns).  These tests write NaN, +Inf
and -Inf, through pa_pool_import, into every pool position that no batch
entry's context covers, run the attention call again, and compare every
output row with the oracle, which only ever reads positions below each
context length (kgptalkie "Day 28: PagedAttention / vLLM", "Follow One Token
Address": the kernel scores only the keys its request's table and length
name).
"""
import numpy as np
import pytest
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import runtime, workloads as wls

from gpu_common import run_library, tol

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


def _uncovered(tables, lens, num_blocks, block_size):
    """bool [num_blocks, block_size]: True where no batch entry's context reaches."""
    covered = np.zeros((num_blocks, block_size), dtype=bool)
    for s in range(tables.shape[0]):
        L = int(lens[s])
        if L <= 0:
            continue
        pos = np.arange(L)
        blk = tables[s, pos // block_size]
        covered[blk, pos % block_size] = True
    return ~covered


def _plant(pool, tables, lens):
    """Write NaN / +Inf / -Inf (cycling) into every uncovered position of K and
    V; returns the number of positions written."""
    k, v = pool.export()                       # K [nb][Hkv][B][D], V [nb][Hkv][D][B]
    torch.cuda.synchronize()
    mask = _uncovered(np.asarray(tables), np.asarray(lens), pool.num_blocks, pool.block_size)
    idx_b, idx_o = np.nonzero(mask)
    if len(idx_b) == 0:
        return 0
    ib = torch.as_tensor(idx_b, device=k.device)
    io = torch.as_tensor(idx_o, device=k.device)
    if pool.fp8:
        # e4m3 has no infinity: its NaN codes are S.1111.111
        bad = torch.tensor([0x7F, 0xFF], dtype=torch.uint8, device=k.device)
        kfill = bad[torch.arange(k.shape[1] * k.shape[3], device=k.device) % 2]
    else:
        bad = torch.tensor([float("nan"), float("inf"), float("-inf")], device=k.device)
        kfill = bad[torch.arange(k.shape[1] * k.shape[3], device=k.device) % 3].to(k.dtype)
    kfill = kfill.view(k.shape[1], k.shape[3])
    k[ib, :, io, :] = kfill.unsqueeze(0).expand(len(idx_b), -1, -1)
    v[ib, :, :, io] = kfill.unsqueeze(0).expand(len(idx_b), -1, -1)
    pool.import_(k, v)
    torch.cuda.synchronize()
    return len(idx_b)


def _decode_case(wl, shared):
    values = wls.generate_values(wl, "cuda")
    pool, bm, _, step = run_library(wl, values, shared=shared)
    assert pool.get_error() == 0
    n = _plant(pool, step.block_tables.cpu().numpy(), step.context_lens.cpu().numpy())
    assert n > 0
    step.out.fill_(float("nan"))
    step.decode()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    got = step.out.double().cpu().numpy()
    assert np.isfinite(got).all(), "a planted non-finite value reached the output"
    st = orp.replay(wl, values)
    ref = orp.attention(wl, values, st, threads=4)
    err = np.abs(got - ref).max()
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"
    return step


DECODE = [
    ("decode", dict(lengths=[1, 15, 17, 33, 100, 250], **D128)),
    ("decode", dict(lengths=[3, 31, 70], dtype="fp8", **D128)),
    ("decode", dict(lengths=[3, 31, 70], dtype="f32", **D128)),
    ("decode", dict(lengths=[5, 19, 41], block_size=32, **D128)),
    ("long", dict(num_seqs=2, min_len=3001, max_len=5003, **D128)),
    ("mixed", dict(num_seqs=24, median=60, min_len=1, max_len=400, prefix_min=20, prefix_max=90,
                   num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="fp8")),
]


@pytest.mark.parametrize("name,kw", DECODE, ids=[f"{n}{i}" for i, (n, _) in enumerate(DECODE)])
def test_decode_ignores_stale_nonfinite(name, kw):
    _decode_case(wls.make_workload(name, **kw), shared=False)


@pytest.mark.parametrize("prefix_len", [41, 16 * 21 + 3, 16 * 64 + 5])
@pytest.mark.parametrize("kernel", ["tcgen05", "mma_sync", "fp8_tcgen05", "fp8_mma_sync"])
def test_shared_prefix_ignores_stale_nonfinite(prefix_len, kernel):
    """pa_decode_shared: shared spans of 2, 21 and 64 full blocks (steps of 64
    tokens that leave 2, 3 and 0 block slots unloaded at the span's end), on
    both kernel forms, for bf16 pools and for fp8 pools (their NaN codes
    planted)."""
    fp8 = kernel.startswith("fp8")
    wl = wls.make_workload("prefix", num_seqs=6, prefix_len=prefix_len, suffix_min=1,
                           suffix_max=40, **D128, **({"dtype": "fp8"} if fp8 else {}))
    values = wls.generate_values(wl, "cuda")
    pool, bm, _ = runtime.replay_setup(wl, values, "cuda")
    pool.set_option("shared_kernel", 1 if kernel.endswith("mma_sync") else 0)
    step = runtime.prepare_step(wl, values, pool, bm, shared=True)
    assert step.sharing()
    step.run()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    n = _plant(pool, step.block_tables.cpu().numpy(), step.context_lens.cpu().numpy())
    assert n > 0
    step.out.fill_(float("nan"))
    step.decode()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    got = step.out.double().cpu().numpy()
    assert np.isfinite(got).all(), "a planted non-finite value reached the output"
    st = orp.replay(wl, values)
    ref = orp.attention(wl, values, st, threads=4)
    err = np.abs(got - ref).max()
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"


PREFILL = [
    dict(lengths=[5, 0, 37], chunks=[20, 13, 70], **D128),
    dict(lengths=[0, 250], chunks=[129, 3], **D128),
    dict(lengths=[17, 40], chunks=[1, 31], num_q_heads=64, num_kv_heads=8, head_dim=128),
    dict(lengths=[9, 0], chunks=[23, 40], num_q_heads=16, num_kv_heads=4, head_dim=64),
    dict(lengths=[7, 30], chunks=[25, 3], num_q_heads=32, num_kv_heads=8, head_dim=128,
         dtype="fp8"),
]


@pytest.mark.parametrize("kw", PREFILL, ids=[f"case{i}" for i in range(len(PREFILL))])
@pytest.mark.parametrize("kernel", ["tcgen05", "mma_sync"])
def test_prefill_ignores_stale_nonfinite(kw, kernel):
    """pa_prefill, both kernels: NaN/Inf in each sequence's last block past its
    length (after the chunk's append) and in every block no sequence uses."""
    wl = wls.make_workload("prefill", **kw)
    values = wls.generate_values(wl, "cuda")
    pool, bm, _ = runtime.replay_setup(wl, values, "cuda")
    pool.set_option("prefill_kernel", 1 if kernel == "mma_sync" else 0)
    step = runtime.prepare_prefill(wl, values, pool, bm)
    step.run()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    n = _plant(pool, step.block_tables.cpu().numpy(), step.context_lens.cpu().numpy())
    assert n > 0
    step.out.fill_(float("nan"))
    step.attend()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    got = step.out.double().cpu().numpy()
    assert np.isfinite(got).all(), "a planted non-finite value reached the output"
    st = orp.replay(wl, values)
    ref = orp.prefill_attention(wl, values, st, threads=4)
    err = np.abs(got - ref).max()
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"


def test_pool_options_round_trip_and_reject_bad_values():
    from paged_kv_cache_253_gb300._lib import PagedAttnError
    pool = runtime.KVPool(4, 16, 2, 128, "bf16", "cuda")
    assert pool.get_option("partition_cap") == -1
    assert pool.get_option("shared_kernel") == 0
    assert pool.get_option("prefill_kernel") == 0
    pool.set_option("partition_cap", 512)
    pool.set_option("prefill_kernel", 1)
    assert pool.get_option("partition_cap") == 512
    assert pool.get_option("prefill_kernel") == 1
    for name, bad in (("partition_cap", -2), ("shared_kernel", 2), ("prefill_kernel", -1)):
        with pytest.raises(PagedAttnError):
            pool.set_option(name, bad)
    assert pool.get_option("partition_cap") == 512
