"""pa_decode_noalloc: decode for callers that cannot let the library allocate.

Some callers own all device memory through their own allocator, or cannot
afford cudaMalloc's device-wide synchronisation inside a serving loop.  For
them the library offers a decode entry point whose scratch lives in a fixed
array inside the library image.  These tests call it through the C ABI and
check its output against pa_decode's on the same inputs, twice in a row (the
second call finds the array holding the first call's bytes), and that a batch
too large for the array is refused before anything runs.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import _lib as L
from paged_kv_cache_253_gb300 import runtime
from paged_kv_cache_253_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

TOL = {"bf16": 5e-3, "f32": 1e-5}   # max-abs tolerances of the parity tests


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(pool, q, tables, lens, scale, out):
    return L.pa_decode_noalloc(pool.handle, _p(q), q.shape[0], q.shape[1], _p(tables),
                               tables.shape[1], _p(lens), scale, _p(out), L.PA_F32,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _two_calls(wl, sample=None):
    """pa_decode's output, then two pa_decode_noalloc calls in a row, each
    compared with it and with the float64 oracle (on `sample` sequences, or
    all of them)."""
    values = wls.generate_values(wl, "cpu")
    pool, bm, _ = runtime.replay_setup(wl, values, "cuda")
    step = runtime.prepare_step(wl, values, pool, bm)
    step.run()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    ref = step.out.clone()
    st = orp.replay(wl, values)
    seqs = sample if sample is not None else list(range(wl.num_seqs))
    oracle = orp.attention(wl, values, st, seqs=seqs, threads=8)
    tol = TOL[wl.dtype]
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(pool, step.q, step.block_tables, step.context_lens, step.scale, out)
        assert rc == 0, L.pa_error_string(rc)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        err = (out - ref).abs().max().item()
        assert err <= tol, f"call {call}: max-abs {err:.3g} against pa_decode"
        got = out.double().cpu().numpy()[seqs]
        err_o = abs(got - oracle).max()
        assert err_o <= tol, f"call {call}: max-abs {err_o:.3g} against the oracle"


def test_noalloc_matches_pa_decode_on_two_calls():
    # lengths up to 6000 so sequences split into several partitions whose
    # partials live in the fixed array
    _two_calls(wls.make_workload("decode", num_seqs=8, min_len=1, max_len=6000, num_q_heads=32,
                                 num_kv_heads=8, head_dim=128))


def test_noalloc_batch_that_only_just_fits_the_array():
    # 1650 sequences x 8 KV heads at G 4, head_dim 128: on a 152-SM GPU the
    # array holds fewer partial slots than the plan would like (16,131 of
    # 16,848) but more than it needs (15,024), so the call gives the kernel the
    # smaller capacity and the partitions grow to fit it
    _two_calls(wls.make_workload("decode", num_seqs=1650, min_len=1, max_len=200,
                                 num_q_heads=32, num_kv_heads=8, head_dim=128),
               sample=[0, 1, 777, 1648, 1649])


def test_noalloc_fp32_pool():
    # the fp32 CUDA-core kernel, whose partial count follows the table width
    _two_calls(wls.make_workload("decode", num_seqs=5, min_len=1, max_len=900, dtype="f32",
                                 num_q_heads=16, num_kv_heads=4, head_dim=64))


def test_noalloc_refuses_a_batch_beyond_its_scratch():
    S, hq, hkv, d = 16384, 32, 8, 128
    pool = runtime.KVPool(4, 16, hkv, d, "bf16", "cuda")
    # real buffers of the claimed size, so nothing could read outside them
    q = torch.zeros((S, hq, d), dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros((S, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(S, dtype=torch.int32, device="cuda")
    out = torch.zeros((S, hq, d), dtype=torch.float32, device="cuda")
    rc = _noalloc(pool, q, tables, lens, 1.0, out)
    assert rc == L.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert pool.get_error() == 0
