"""Retained prefix blocks on the GPU: with retention on, a request admitted
after another one finished takes back that request's full prefix blocks from
the hash table, and the decode reads their keys and values from the pool as
the first request left them; only the new tokens are appended.  Compared with
the oracle's contiguous attention over the expected history."""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from paged_kv_cache_253_gb300.api import BlockManager, KVPool

pytestmark = pytest.mark.gpu

B, HKV, HQ, D = 16, 8, 32, 128


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_retained_prefix_blocks_are_reused_with_their_contents():
    rng = np.random.default_rng(7)
    g = torch.Generator().manual_seed(7)
    nb = 64
    bm = BlockManager(nb, B, rng.permutation(nb))
    bm.set_retention(True)
    pool = KVPool(nb, B, HKV, D, "bf16", "cuda")

    prompt = rng.integers(0, 1000, size=5 * B + 3).tolist()
    a, cached = bm.add_request(prompt)
    assert cached == 0
    slots_a = [bm.append_slot(a, t)[0] for t in prompt]
    ka = torch.randn(len(prompt), HKV, D, generator=g).to(torch.bfloat16)
    va = torch.randn(len(prompt), HKV, D, generator=g).to(torch.bfloat16)
    pool.append_kv(ka.cuda(), va.cuda(), torch.tensor(slots_a, dtype=torch.int64, device="cuda"))
    table_a = bm.block_table(a)
    bm.free_request(a)
    assert bm.num_evictable() == 5                    # the five full blocks stay cached

    own = rng.integers(0, 1000, size=7).tolist()
    b, cached = bm.add_request(prompt[:5 * B] + own)
    assert cached == 5 * B and bm.block_table(b)[:5] == table_a[:5]
    assert bm.num_evictable() == 0
    slots_b = [bm.append_slot(b, t)[0] for t in own]
    kb = torch.randn(len(own), HKV, D, generator=g).to(torch.bfloat16)
    vb = torch.randn(len(own), HKV, D, generator=g).to(torch.bfloat16)
    pool.append_kv(kb.cuda(), vb.cuda(), torch.tensor(slots_b, dtype=torch.int64, device="cuda"))

    tables, lens = bm.batch_tables([b])
    q = torch.randn(1, HQ, D, generator=g).to(torch.bfloat16)
    out = pool.decode(q.cuda(), torch.as_tensor(tables, device="cuda"),
                      torch.as_tensor(lens, device="cuda"), 1.0 / np.sqrt(D))
    torch.cuda.synchronize()
    assert pool.get_error() == 0

    kseq = _bits(torch.cat([ka[:5 * B], kb]))
    vseq = _bits(torch.cat([va[:5 * B], vb]))
    ref = oatt.contiguous_decode(q.double().numpy(), [kseq], [vseq], 1.0 / np.sqrt(D), HKV)
    err = np.abs(out.double().cpu().numpy() - ref).max()
    assert err <= 5e-3, f"max-abs {err:.3g}"

