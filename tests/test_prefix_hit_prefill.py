"""A prefix-cache hit skips the prefill of the cached span (zenaique prefix-
sharing answer and kgptalkie "Prefix Sharing Is a Natural Extension": a hit on
the chained block hash reuses the block, and that span needs no prefill).

Request a prefills a whole prompt and finishes; with retention on its full
blocks stay registered.  Request b, admitted with the same leading tokens and
its own tail, gets those blocks back from the hash table and prefills only
its tail: each tail query must see a's keys and values for the shared span
and b's own for the tail, exactly as contiguous causal attention over the
whole of b's history does.

The flow runs twice: on the CPU with the C++ block manager and the oracle's
pool (checks the flow itself), and on the GPU through the library.
"""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import kvcache as okv
from oracle import prefill as opf

B, HKV, HQ, D = 16, 8, 32, 128
NB = 64
SCALE = 1.0 / np.sqrt(D)


def _draw(rng, n, heads):
    """bf16 values (as raw bits) of n rows."""
    x = rng.standard_normal((n, heads, D)).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)      # truncation to bf16 bits


def _reference(q_bits, k_hist, v_hist, start):
    """Contiguous causal attention: query row i sits at position start + i."""
    q = oatt.bf16_bits_to_f32(q_bits)
    n = q.shape[0]
    ks = [k_hist[:start + i + 1] for i in range(n)]
    vs = [v_hist[:start + i + 1] for i in range(n)]
    return oatt.contiguous_decode(q, ks, vs, SCALE, HKV)


class _OraclePool:
    """The oracle's bit-level pool behind the same three calls."""

    def __init__(self):
        self.k = np.zeros((NB, HKV, B, D), np.uint16)
        self.v = np.zeros((NB, HKV, B, D), np.uint16)

    def append(self, k, v, slots):
        okv.append_kv(self.k, self.v, k, v, np.asarray(slots, np.int64))

    def prefill(self, q, n, tables, lens):
        cu = np.array([0, n], np.int32)
        return opf.paged_prefill(oatt.bf16_bits_to_f32(q), self.k, self.v, tables, cu, lens,
                                 SCALE, HKV)


class _GpuPool:
    def __init__(self):
        import torch
        from paged_kv_cache_253_gb300.api import KVPool
        self.torch = torch
        self.pool = KVPool(NB, B, HKV, D, "bf16", "cuda")

    def _t(self, bits):
        return self.torch.from_numpy(bits.view(np.int16)).view(self.torch.bfloat16).cuda()

    def append(self, k, v, slots):
        t = self.torch
        self.pool.append_kv(self._t(k), self._t(v), t.as_tensor(np.asarray(slots, np.int64)).cuda())

    def prefill(self, q, n, tables, lens):
        t = self.torch
        out = self.pool.prefill(self._t(q), t.tensor([0, n], dtype=t.int32).cuda(),
                                t.as_tensor(tables).cuda(), t.as_tensor(lens).cuda(), SCALE,
                                max_q_len=n)
        t.cuda.synchronize()
        assert self.pool.get_error() == 0
        return out.double().cpu().numpy()


def _flow(pool):
    from paged_kv_cache_253_gb300.api import BlockManager
    rng = np.random.default_rng(2531)
    bm = BlockManager(NB, B, rng.permutation(NB))
    bm.set_retention(True)
    shared, tail_a, tail_b = 5 * B, 7, 30
    prompt = rng.integers(0, 1000, size=shared + tail_a).tolist()

    # request a: the whole prompt is prefilled
    a, cached = bm.add_request(prompt)
    assert cached == 0
    slots, pairs = bm.append_slots([a] * len(prompt), prompt)
    assert len(pairs) == 0
    k_a, v_a = _draw(rng, len(prompt), HKV), _draw(rng, len(prompt), HKV)
    pool.append(k_a, v_a, slots)
    tables, lens = bm.batch_tables([a])
    q_a = _draw(rng, len(prompt), HQ)
    out_a = pool.prefill(q_a, len(prompt), tables, lens)
    ref_a = _reference(q_a, oatt.bf16_bits_to_f32(k_a), oatt.bf16_bits_to_f32(v_a), 0)
    err_a = float(np.abs(out_a - ref_a).max())
    table_a = bm.block_table(a)
    bm.free_request(a)
    assert bm.num_evictable() == shared // B

    # request b: the shared span hits the cache; only b's tail is prefilled
    own = rng.integers(1000, 2000, size=tail_b).tolist()
    b, cached = bm.add_request(prompt[:shared] + own)
    assert cached == shared and bm.block_table(b)[:shared // B] == table_a[:shared // B]
    slots, pairs = bm.append_slots([b] * tail_b, own)
    assert len(pairs) == 0                       # the tail starts a fresh block
    k_b, v_b = _draw(rng, tail_b, HKV), _draw(rng, tail_b, HKV)
    pool.append(k_b, v_b, slots)
    tables, lens = bm.batch_tables([b])
    assert lens.tolist() == [shared + tail_b]
    q_b = _draw(rng, tail_b, HQ)
    out_b = pool.prefill(q_b, tail_b, tables, lens)
    k_hist = oatt.bf16_bits_to_f32(np.concatenate([k_a[:shared], k_b]))
    v_hist = oatt.bf16_bits_to_f32(np.concatenate([v_a[:shared], v_b]))
    ref_b = _reference(q_b, k_hist, v_hist, shared)
    return err_a, float(np.abs(out_b - ref_b).max())


def test_prefix_hit_prefill_flow_with_the_oracle_pool():
    pytest.importorskip("torch")
    from paged_kv_cache_253_gb300 import build
    build.build()
    err_a, err_b = _flow(_OraclePool())
    assert err_a < 1e-12 and err_b < 1e-12


@pytest.mark.gpu
def test_prefix_hit_prefill_on_the_gpu():
    err_a, err_b = _flow(_GpuPool())
    assert err_a <= 5e-3 and err_b <= 5e-3, (err_a, err_b)
