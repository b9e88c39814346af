"""GPU parity of paged (chunked) prefill against the oracle.

Each batch entry appends a chunk of new tokens (copy-on-write and slots from
the C++ block manager, keys/values through pa_append_kv) and pa_prefill runs
the chunk's queries: each attends to its request's cached prefix and causally
to the chunk up to itself.  Bookkeeping and pools bit-exact; attention
max-abs <= BF16_TOL (bf16 q/K/V, fp32 accumulation) against the float64
oracle, at small sizes with ragged chunks (1, 15, 16, 17, 33 tokens; tile
boundaries of 64 rows) and on sampled sequences of the full workload.
"""
import numpy as np
import pytest
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import runtime, workloads as wls
from paged_kv_cache_253_gb300._lib import PagedAttnError

from gpu_common import BF16_TOL, assert_pools_equal

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


_FORM = {"prefill_kernel": 0}      # set by the `form` fixture


def _run(wl, values, out_dtype=torch.float32):
    pool, bm, setup_pairs = runtime.replay_setup(wl, values, "cuda")
    pool.set_option("prefill_kernel", _FORM["prefill_kernel"])
    step = runtime.prepare_prefill(wl, values, pool, bm, out_dtype=out_dtype)
    step.run()
    torch.cuda.synchronize()
    return pool, setup_pairs, step


def _check(wl, values, seqs=None, threads=1, out_dtype=torch.float32):
    pool, setup_pairs, step = _run(wl, values, out_dtype)
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert setup_pairs == st.setup_pairs
    assert step.slots.cpu().numpy().tolist() == st.step_slots.tolist()
    assert np.array_equal(step.block_tables.cpu().numpy(), st.block_tables)
    assert np.array_equal(step.context_lens.cpu().numpy(), st.context_lens)
    assert np.array_equal(step.cu_seqlens_q.cpu().numpy(), st.cu_seqlens_q)
    assert_pools_equal(pool, st)
    ref = orp.prefill_attention(wl, values, st, seqs=seqs, threads=threads)
    got = step.out.double().cpu().numpy()
    if seqs is not None:
        cu = st.cu_seqlens_q
        got = got[np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])]
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= BF16_TOL, f"max-abs {err:.3g} > {BF16_TOL}"
    return err, step


SMALL = [
    dict(lengths=[0, 3, 40, 16], chunks=[1, 15, 16, 17], **D128),
    dict(lengths=[5, 0, 100], chunks=[33, 64, 47], **D128),
    dict(lengths=[0, 21], chunks=[130, 9], num_q_heads=64, num_kv_heads=8, head_dim=128),    # G = 8
    dict(lengths=[7, 0], chunks=[70, 3], num_q_heads=8, num_kv_heads=8, head_dim=128),       # G = 1
    dict(lengths=[19, 2], chunks=[40, 23], num_q_heads=10, num_kv_heads=2, head_dim=128),    # G = 5
    dict(lengths=[33, 0], chunks=[50, 17], num_q_heads=16, num_kv_heads=4, head_dim=64),
    dict(lengths=[12, 30], chunks=[29, 8], num_q_heads=8, num_kv_heads=2, head_dim=256),
    dict(lengths=[45, 0, 3], chunks=[20, 33, 1], block_size=32, **D128),
    dict(num_seqs=4, min_len=0, max_len=600, chunk_min=1, chunk_max=200, **D128),
]


@pytest.fixture(params=["default", "mma_sync"])
def form(request):
    """The default dispatch (tcgen05 for bf16 pools of 16-token blocks and
    head_dim 128, mma.sync otherwise) and the mma.sync kernel selected through
    the pool's PA_OPT_PREFILL_KERNEL option."""
    _FORM["prefill_kernel"] = 1 if request.param == "mma_sync" else 0
    yield request.param
    _FORM["prefill_kernel"] = 0


@pytest.mark.parametrize("kw", SMALL, ids=[f"case{i}" for i in range(len(SMALL))])
def test_small_parity(kw, form):
    wl = wls.make_workload("prefill", **kw)
    values = wls.generate_values(wl, "cuda")
    err, _ = _check(wl, values)
    print(f"prefill [{form}] {kw}: max-abs {err:.3g}")


def test_bf16_output_is_the_fp32_output_rounded(form):
    wl = wls.make_workload("prefill", lengths=[9, 0], chunks=[20, 37], **D128)
    values = wls.generate_values(wl, "cuda")
    _, step = _check(wl, values)
    out16 = step.pool.prefill(step.q, step.cu_seqlens_q, step.block_tables, step.context_lens,
                              step.scale, max_q_len=step.max_q_len, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out16, step.out.to(torch.bfloat16))


def test_two_chunks_equal_one(form):
    """A prompt prefilled as one chunk, and as two chunks with the second
    after the first's append, gives the second chunk's rows the same outputs
    (up to fp32 summation order: the tiles differ)."""
    prompt, first = 150, 61
    wl1 = wls.make_workload("prefill", lengths=[0], chunks=[prompt], **D128)
    v1 = wls.generate_values(wl1, "cuda")
    _, _, s1 = _run(wl1, v1)
    # the same tokens and values, the first 61 of them cached beforehand
    wl2 = wls.make_workload("prefill", lengths=[first], chunks=[prompt - first], **D128)
    v2 = {"q": v1["q"][first:], "new_k": v1["new_k"][first:], "new_v": v1["new_v"][first:],
          "hist_k": v1["new_k"][:first], "hist_v": v1["new_v"][:first]}
    _, _, s2 = _run(wl2, v2)
    a = s1.out[first:].double().cpu()
    b = s2.out.double().cpu()
    assert (a - b).abs().max().item() <= 1e-5


def test_device_errors_are_recorded_not_faulted(form):
    wl = wls.make_workload("prefill", lengths=[10, 4], chunks=[8, 6], **D128)
    values = wls.generate_values(wl, "cuda")
    pool, _, step = _run(wl, values)
    assert pool.get_error() == 0
    # a chunk longer than max_q_len
    pool.prefill(step.q, step.cu_seqlens_q, step.block_tables, step.context_lens, step.scale,
                 max_q_len=4, out=step.out)
    assert pool.get_error() == -1
    # a chunk longer than its context
    bad_lens = step.context_lens.clone()
    bad_lens[1] = 3
    pool.prefill(step.q, step.cu_seqlens_q, step.block_tables, bad_lens, step.scale,
                 max_q_len=8, out=step.out)
    assert pool.get_error() == -1
    # a block id outside the pool
    bad_tables = step.block_tables.clone()
    bad_tables[0, 0] = wl.num_blocks + 5
    pool.prefill(step.q, step.cu_seqlens_q, bad_tables, step.context_lens, step.scale,
                 max_q_len=8, out=step.out)
    assert pool.get_error() == -5
    # host checks: the binding's dtype check, and the library's (an fp32 pool)
    with pytest.raises(TypeError):
        pool.prefill(step.q.float(), step.cu_seqlens_q, step.block_tables, step.context_lens,
                     step.scale, max_q_len=8)
    from paged_kv_cache_253_gb300.api import KVPool
    pool32 = KVPool(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, "f32", "cuda")
    with pytest.raises(PagedAttnError) as e:
        pool32.prefill(step.q.float(), step.cu_seqlens_q, step.block_tables, step.context_lens,
                       step.scale, max_q_len=8)
    assert e.value.code == -2
    assert pool.get_error() == 0


def test_full_size_parity(form):
    """The prefill workload (16 sequences, cached prefixes up to 4096, chunks of
    128..512) at full size: bookkeeping and pools bit-exact, attention on every
    row of sampled sequences."""
    wl = wls.make_workload("prefill")
    values = wls.generate_values(wl, "cuda")
    seqs = [0, 7, wl.num_seqs - 1]
    err, _ = _check(wl, values, seqs=seqs, threads=16)
    print(f"prefill [{form}] full size: max-abs over sequences {seqs}: {err:.3g}")
