"""Decode schedule regions (GPU).

The split pass chooses its partition length on the device from the batch's
total length: the item target is whole waves of one item per resident CTA
(one wave per MiB of cache each CTA reads, at most twelve items per SM), and
on fp8 pools the smallest partition grows from 64 towards 256 tokens while two
items per SM remain, which also decides whether the guided tail (shorter
partitions for the last quarter of the tokens) runs.  Each region of that
choice changes how a sequence is cut into partials and merged, so each gets a
parity case against the oracle here: the result must not depend on where a
sequence is cut (kgptalkie "Day 28: PagedAttention / vLLM", "Follow One Token
Address": each query scores exactly the keys its table and length name).

`_plan` restates the rule on the host only to check that a case lands in the
region it is meant to cover (152 SMs; 4 resident CTAs per SM for fp8 pools and
3 for bf16 ones at D = 128).
"""

import numpy as np
import pytest
import torch

from oracle import replay as orp
from paged_kv_cache_253_gb300 import runtime, workloads as wls

from gpu_common import assert_pools_equal, tol

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


def _plan(lens, hkv, block, fp8, sms):
    total = int(sum(int(x) for x in lens))
    grid = sms * (4 if fp8 else 3)
    wave_tokens = (1 << 20) // (2 * 128 * (1 if fp8 else 2))
    waves = max(1, -(-total * hkv // (grid * wave_tokens)))
    target = min(sms * 12, waves * grid)
    need = -(-total * hkv // target)
    need = -(-need // block) * block
    pmin = 64
    if fp8:
        cap = total * hkv // (2 * sms) // block * block
        pmin = max(64, min(256, cap))
    pt = max(need, pmin)
    pts = max(pmin, -(-(pt // 4) // block) * block)
    return dict(waves=waves, pmin=pmin, pt=pt, tail=pts < pt and pts >= 256)


def _run(wl, values, seqs, partition_cap=None):
    pool, bm, _ = runtime.replay_setup(wl, values, "cuda")
    if partition_cap is not None:
        pool.set_option("partition_cap", partition_cap)
    step = runtime.prepare_step(wl, values, pool, bm)
    step.run()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert_pools_equal(pool, st)
    ref = orp.attention(wl, values, st, seqs=seqs, threads=8)
    got = step.out.double().cpu().numpy()[np.asarray(seqs)]
    err = np.abs(got - ref).max()
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"
    return st, err


CASES = [
    # fp8, a few thousand tokens: the smallest partition between 64 and 256
    ("soft_min", "decode", dict(num_seqs=4, min_len=500, max_len=2000, dtype="fp8", **D128), None,
     lambda r: 64 < r["pmin"] < 256 and r["waves"] == 1),
    # fp8, tens of thousands of tokens: smallest partition 256, guided tail on
    ("tail", "decode", dict(num_seqs=24, min_len=500, max_len=2000, dtype="fp8", **D128), None,
     lambda r: r["pmin"] == 256 and r["tail"] and r["waves"] == 1),
    # fp8, a few hundred thousand tokens: two waves of items
    ("fp8_two_waves", "long", dict(num_seqs=4, min_len=80000, max_len=150000, dtype="fp8", **D128),
     None, lambda r: r["waves"] == 2),
    # bf16: two waves of items
    ("bf16_two_waves", "decode", dict(num_seqs=16, min_len=8000, max_len=16000, **D128), None,
     lambda r: r["waves"] == 2),
    # fp8 with a 64-token partition cap: the smallest partition stays at the cap
    ("cap_below_min", "decode", dict(num_seqs=24, min_len=500, max_len=2000, dtype="fp8", **D128), 64,
     lambda r: r["pmin"] == 256),
]


@pytest.mark.parametrize("tag,name,kw,cap,region", CASES, ids=[c[0] for c in CASES])
def test_schedule_region_parity(tag, name, kw, cap, region):
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cuda")
    S = wl.num_seqs
    seqs = sorted({0, S - 1} | set(np.random.default_rng(wl.seed).choice(S, size=min(4, S),
                                                                         replace=False).tolist()))
    st, err = _run(wl, values, seqs, partition_cap=cap)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    r = _plan(st.context_lens, wl.num_kv_heads, wl.block_size, wl.dtype == "fp8", sms)
    if sms == 152:
        assert region(r), f"{tag}: the batch lands outside its schedule region: {r}"
    print(f"{tag}: {r}, max-abs {err:.3g} over {len(seqs)} sequences")
