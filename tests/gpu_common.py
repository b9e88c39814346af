"""Helpers for the GPU parity tests: run a workload through the library and
through the oracle, and put the two pools in one layout for comparison."""
import numpy as np
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import runtime, workloads

BF16_TOL = 5e-3     # max-abs, bf16 K/V/Q with fp32 accumulation
F32_TOL = 1e-5      # max-abs, fp32 pool
# fp8 pool, against attention over the codes' exact values: the codes widen
# exactly to f16, bf16 queries to f16 exactly (|q| >= 2^-17), the
# probabilities enter as an f16 pair (hi + remainder, ~22 bits) and every sum
# is fp32 — so fp32 rounding, not the 8-bit storage, sets the error; values
# reach |v_scale * 448| ~ 6.3, hence a bound a few times F32_TOL.
FP8_TOL = 5e-5


def tol(wl):
    return {"f32": F32_TOL, "fp8": FP8_TOL}.get(wl.dtype, BF16_TOL)


def bits(t):
    """Raw element bits of a tensor as numpy (uint16 for bf16, float32 kept)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run_library(wl, values, out_dtype=torch.float32, shared=True, fused=True):
    pool, bm, setup_pairs = runtime.replay_setup(wl, values, "cuda")
    step = runtime.prepare_step(wl, values, pool, bm, out_dtype=out_dtype, shared=shared,
                                fused=fused)
    step.run()
    torch.cuda.synchronize()
    return pool, bm, setup_pairs, step


def pool_in_oracle_layout(pool):
    """(K, V) of the library's pool as numpy bits in [nb][Hkv][B][D] order:
    the library keeps V transposed per tile ([nb][Hkv][D][B])."""
    k, v = pool.export()
    torch.cuda.synchronize()
    return bits(k), bits(v.transpose(2, 3).contiguous())


def assert_pools_equal(pool, st, chunk=4096):
    k, v = pool.export()
    torch.cuda.synchronize()
    nb = k.shape[0]
    for lo in range(0, nb, chunk):
        hi = min(nb, lo + chunk)
        kb = bits(k[lo:hi])
        vb = bits(v[lo:hi].transpose(2, 3).contiguous())
        assert np.array_equal(kb.view(np.uint8), st.k_pool[lo:hi].view(np.uint8)), \
            f"K differs in blocks [{lo},{hi})"
        assert np.array_equal(vb.view(np.uint8), st.v_pool[lo:hi].view(np.uint8)), \
            f"V differs in blocks [{lo},{hi})"
