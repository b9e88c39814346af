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

from paged_kv_cache_253_gb300 import _lib as L
from paged_kv_cache_253_gb300 import runtime
from paged_kv_cache_253_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

TOL = 5e-3      # max-abs tolerance of the bf16 parity tests


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(pool, q, tables, lens, scale, out):
    return L.pa_decode_noalloc(pool.handle, _p(q), q.shape[0], q.shape[1], _p(tables),
                               tables.shape[1], _p(lens), scale, _p(out), L.PA_F32,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_pa_decode_on_two_calls():
    # lengths up to 6000 so sequences split into several partitions and the
    # arrival counters in the fixed array are exercised
    wl = wls.make_workload("decode", num_seqs=8, min_len=1, max_len=6000, num_q_heads=32,
                           num_kv_heads=8, head_dim=128)
    values = wls.generate_values(wl, "cpu")
    pool, bm, _ = runtime.replay_setup(wl, values, "cuda")
    step = runtime.prepare_step(wl, values, pool, bm)
    step.run()
    torch.cuda.synchronize()
    ref = step.out.clone()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(pool, step.q, step.block_tables, step.context_lens, step.scale, out)
        assert rc == 0, L.pa_error_string(rc)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        err = (out - ref).abs().max().item()
        assert err <= TOL, f"call {call}: max-abs {err:.3g}"


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
