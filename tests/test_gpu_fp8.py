"""GPU parity of the fp8 (e4m3) KV pool against the oracle.

* append: every stored code equals the oracle's quantization of the bf16
  input under the pool's K or V scale — bit-exact, rounding ties, subnormals,
  saturation and infinities included;
* copy-on-write copies move codes bit for bit (whole replayed workloads);
* attention over the codes' values (code * scale) — max-abs <= FP8_TOL, on
  the tensor-core shapes and on the fp32 CUDA-core kernel, small cases with
  ragged tails and a full-size batch on sampled sequences.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import fp8
from oracle import replay as orp
from paged_kv_cache_253_gb300 import runtime, workloads as wls
from paged_kv_cache_253_gb300._lib import PagedAttnError
from paged_kv_cache_253_gb300.api import KVPool

from gpu_common import FP8_TOL, assert_pools_equal, run_library, tol

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="fp8")


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _awkward_values(g, n, hkv, d, scale):
    """bf16 rows with every rounding case: exact e4m3 midpoints times the scale
    (ties, when the scale is a power of two), subnormal codes, magnitudes just
    above 448 and far beyond it, +-inf, signed zeros."""
    x = torch.randn(n, hkv, d, generator=g) * 2.0
    flat = x.view(-1)
    m = flat.numel()
    idx = torch.randperm(m, generator=g)
    k = m // 16
    mant = torch.randint(0, 8, (k,), generator=g).float()
    expo = torch.randint(-6, 9, (k,), generator=g).float()
    mid = torch.where(expo == -6, (mant + 0.5) * 2.0 ** -9, (8 + mant + 0.5) * torch.exp2(expo - 3))
    flat[idx[:k]] = mid * scale
    flat[idx[k:2 * k]] = torch.rand(k, generator=g) * (2 ** -6) * scale           # subnormal codes
    flat[idx[2 * k:3 * k]] = (448 + torch.rand(k, generator=g) * 40) * scale      # 448 .. 488
    flat[idx[3 * k:4 * k]] = (torch.rand(k, generator=g) + 1) * 600 * scale       # saturate
    flat[idx[4 * k:4 * k + 4]] = torch.tensor([float("inf"), float("-inf"), 0.0, -0.0])
    flat[idx[:4 * k]] *= torch.where(torch.rand(4 * k, generator=g) < 0.5, -1.0, 1.0)
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("d,B,ks,vs", [(128, 16, 0.0173, 0.0141), (64, 32, 2.0 ** -6, 2.0 ** -5),
                                       (96, 8, 0.031, 2.0 ** -4)])
def test_append_codes_are_the_oracles_quantization(d, B, ks, vs):
    g = torch.Generator().manual_seed(31 + d)
    nb, hkv, T = 40, 4, 300
    pool = KVPool(nb, B, hkv, d, "fp8", "cuda")
    pool.set_kv_scales(ks, vs)
    assert pool.kv_scales() == (float(np.float32(ks)), float(np.float32(vs)))
    k = _awkward_values(g, T, hkv, d, ks)
    v = _awkward_values(g, T, hkv, d, vs)
    slots = torch.randperm(nb * B, generator=g)[:T].to(torch.int64)
    slots[::37] = -1                                  # skipped tokens
    pool.append_kv(k.cuda(), v.cuda(), slots.cuda())
    kp, vp = pool.export()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    kp = kp.cpu().numpy()
    vp = vp.cpu().numpy().transpose(0, 1, 3, 2)        # V is stored transposed per tile
    kf = oatt.bf16_bits_to_f32(_bf16_bits(k))
    vf = oatt.bf16_bits_to_f32(_bf16_bits(v))
    want_k = fp8.quantize(kf, ks)
    want_v = fp8.quantize(vf, vs)
    written = np.zeros((nb, B), dtype=bool)
    for t, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        b, o = divmod(s, B)
        written[b, o] = True
        assert np.array_equal(kp[b, :, o, :], want_k[t]), f"K codes of token {t}"
        assert np.array_equal(vp[b, :, o, :], want_v[t]), f"V codes of token {t}"
    assert not kp.transpose(0, 2, 1, 3)[~written].any()   # nothing else was touched
    assert not vp.transpose(0, 2, 1, 3)[~written].any()
    # the cases were all there
    assert (want_k == 0x7E).any() and (want_k == 0xFE).any() and ((want_k & 0x78) == 0).any()


def test_scales_are_checked():
    pool = KVPool(4, 16, 1, 64, "fp8", "cuda")
    for bad in [(0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))]:
        with pytest.raises(PagedAttnError):
            pool.set_kv_scales(*bad)
    bf = KVPool(4, 16, 1, 64, "bf16", "cuda")
    with pytest.raises(PagedAttnError):
        bf.set_kv_scales(1.0, 1.0)


SMALL = [
    ("decode", dict(num_seqs=6, min_len=1, max_len=300, **D128)),
    ("decode", dict(lengths=[0, 1, 15, 16, 17, 33, 250], **D128)),
    ("decode", dict(num_seqs=4, min_len=1, max_len=200, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, dtype="fp8")),                            # G = 8
    ("decode", dict(num_seqs=4, min_len=1, max_len=200, num_q_heads=16, num_kv_heads=4,
                    head_dim=64, dtype="fp8")),
    ("decode", dict(num_seqs=3, min_len=1, max_len=200, num_q_heads=8, num_kv_heads=2,
                    head_dim=256, dtype="fp8")),
    # G = 1, 2, 3 (score columns 4..7 repeat the group's heads and carry the
    # probabilities' remainders into the value product) and G = 5 (no repeat)
    ("decode", dict(num_seqs=4, min_len=1, max_len=300, num_q_heads=8, num_kv_heads=8,
                    head_dim=128, dtype="fp8")),
    ("decode", dict(lengths=[1, 17, 250], num_q_heads=16, num_kv_heads=8, head_dim=128, dtype="fp8")),
    ("decode", dict(num_seqs=4, min_len=1, max_len=300, num_q_heads=12, num_kv_heads=4,
                    head_dim=128, dtype="fp8")),
    ("decode", dict(num_seqs=4, min_len=1, max_len=300, num_q_heads=20, num_kv_heads=4,
                    head_dim=128, dtype="fp8")),
    ("decode", dict(num_seqs=4, min_len=1, max_len=200, block_size=32, **D128)),
    ("decode", dict(num_seqs=4, min_len=1, max_len=100, block_size=8, **D128)),   # fp32 kernel
    ("decode", dict(num_seqs=3, min_len=1, max_len=100, num_q_heads=32, num_kv_heads=2,
                    head_dim=128, dtype="fp8")),                            # G = 16: fp32 kernel
    ("prefix", dict(num_seqs=6, prefix_len=41, suffix_min=1, suffix_max=40, **D128)),
    ("mixed", dict(num_seqs=24, median=60, min_len=1, max_len=400, prefix_min=20,
                   prefix_max=90, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="fp8")),
    ("long", dict(num_seqs=2, min_len=3000, max_len=9000, **D128)),
]


def _check(wl, values, seqs=None, threads=1, shared=True, fused=True):
    pool, bm, setup_pairs, step = run_library(wl, values, shared=shared, fused=fused)
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert setup_pairs == st.setup_pairs
    assert step.slots.cpu().numpy().tolist() == st.step_slots.tolist()
    assert np.array_equal(step.block_tables.cpu().numpy(), st.block_tables)
    assert_pools_equal(pool, st)
    ref = orp.attention(wl, values, st, seqs=seqs, threads=threads)
    got = step.out.double().cpu().numpy()
    if seqs is not None:
        got = got[np.asarray(seqs)]
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= tol(wl), f"max-abs {err:.3g} > {tol(wl)}"
    return err


@pytest.mark.parametrize("name,kw", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_small_parity(name, kw):
    wl = wls.make_workload(name, **kw)
    values = wls.generate_values(wl, "cuda")
    err = _check(wl, values)
    print(f"{wl.name} {kw}: max-abs {err:.3g}")


@pytest.mark.parametrize("kw", [dict(num_seqs=6, min_len=1, max_len=300, **D128),
                                dict(lengths=[1, 16, 17, 33], num_q_heads=16, num_kv_heads=4,
                                     head_dim=64, dtype="fp8"),
                                dict(num_seqs=3, min_len=1, max_len=200, num_q_heads=8,
                                     num_kv_heads=2, head_dim=256, dtype="fp8"),
                                dict(num_seqs=4, min_len=1, max_len=200, block_size=32, **D128)])
def test_append_decode_equals_separate_calls(kw):
    """An fp8 pool's append_decode (the quantizing append fused into the decode
    kernel on the tensor-core shapes) equals the quantizing append then the
    decode: the same codes in the pool, bit for bit, and the same outputs."""
    wl = wls.make_workload("decode", **kw)
    values = wls.generate_values(wl, "cuda")
    outs, pools = [], []
    for fused in (True, False):
        pool, _, _, step = run_library(wl, values, fused=fused)
        assert pool.get_error() == 0
        outs.append(step.out.cpu())
        k, v = pool.export()
        torch.cuda.synchronize()
        pools.append((k.cpu(), v.cpu()))
    assert torch.equal(pools[0][0], pools[1][0]) and torch.equal(pools[0][1], pools[1][1])
    assert torch.equal(outs[0], outs[1])


PREFILL = [
    dict(lengths=[0, 3, 40, 16], chunks=[1, 15, 16, 17], **D128),
    dict(lengths=[5, 0, 100], chunks=[33, 64, 47], **D128),
    dict(lengths=[0, 21], chunks=[130, 9], num_q_heads=64, num_kv_heads=8, head_dim=128,
         dtype="fp8"),                                                      # G = 8
    dict(lengths=[19, 2], chunks=[40, 23], num_q_heads=10, num_kv_heads=2, head_dim=128,
         dtype="fp8"),                                                      # G = 5
    dict(lengths=[33, 0], chunks=[50, 17], num_q_heads=16, num_kv_heads=4, head_dim=64,
         dtype="fp8"),
    dict(lengths=[12, 30], chunks=[29, 8], num_q_heads=8, num_kv_heads=2, head_dim=256,
         dtype="fp8"),
    dict(lengths=[45, 0, 3], chunks=[20, 33, 1], block_size=32, **D128),
]


def _check_prefill(wl, values, seqs=None, threads=1, kernel="tcgen05"):
    pool, bm, setup_pairs = runtime.replay_setup(wl, values, "cuda")
    pool.set_option("prefill_kernel", 1 if kernel == "mma_sync" else 0)
    step = runtime.prepare_prefill(wl, values, pool, bm)
    step.run()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert setup_pairs == st.setup_pairs
    assert step.slots.cpu().numpy().tolist() == st.step_slots.tolist()
    assert np.array_equal(step.block_tables.cpu().numpy(), st.block_tables)
    assert_pools_equal(pool, st)
    ref = orp.prefill_attention(wl, values, st, seqs=seqs, threads=threads)
    got = step.out.double().cpu().numpy()
    if seqs is not None:
        cu = st.cu_seqlens_q
        got = got[np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])]
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= FP8_TOL, f"max-abs {err:.3g} > {FP8_TOL}"
    return err


@pytest.mark.parametrize("kernel", ["tcgen05", "mma_sync"])
@pytest.mark.parametrize("kw", PREFILL, ids=[f"case{i}" for i in range(len(PREFILL))])
def test_prefill_parity(kw, kernel):
    """Chunked prefill over an fp8 pool: the chunk's codes (quantizing append)
    bit-exact, every query row within FP8_TOL of float64 attention over the
    codes' values; the tcgen05 kernel (codes widened to f16 in shared memory,
    head_dim 128) and the mma.sync form (the other shapes run it either way)."""
    wl = wls.make_workload("prefill", **kw)
    values = wls.generate_values(wl, "cuda")
    err = _check_prefill(wl, values, kernel=kernel)
    print(f"prefill fp8 {kw} {kernel}: max-abs {err:.3g}")


@pytest.mark.parametrize("kernel", ["tcgen05", "mma_sync"])
def test_prefill_full_size_parity(kernel):
    """The prefill workload (16 sequences, cached prefixes up to 4096, chunks of
    128..512) on an fp8 pool: codes bit-exact, attention on sampled sequences."""
    wl = wls.make_workload("prefill", dtype="fp8")
    values = wls.generate_values(wl, "cuda")
    seqs = [0, 7, wl.num_seqs - 1]
    err = _check_prefill(wl, values, seqs=seqs, threads=16, kernel=kernel)
    print(f"prefill fp8 full size ({kernel}): max-abs over sequences {seqs}: {err:.3g}")


def test_full_size_parity():
    """The decode batch at full size (64 sequences of 128..2048 tokens) on an
    fp8 pool: every code bit-exact, attention on sampled sequences."""
    wl = wls.make_workload("decode", dtype="fp8")
    values = wls.generate_values(wl, "cuda")
    rng = np.random.default_rng(wl.seed)
    seqs = sorted(set(rng.choice(wl.num_seqs, size=12, replace=False).tolist()) | {0, wl.num_seqs - 1})
    err = _check(wl, values, seqs=seqs, threads=8)
    print(f"decode fp8 full size: max-abs over {len(seqs)} sequences {err:.3g} (tol {FP8_TOL})")


SHARED = [
    dict(num_seqs=6, prefix_len=300, suffix_min=1, suffix_max=40, **D128),               # G = 4
    dict(num_seqs=70, prefix_len=1100, suffix_min=0, suffix_max=30, **D128),             # 2 chunks, 3 tiles
    dict(num_seqs=9, prefix_len=700, suffix_min=5, suffix_max=60, num_q_heads=64, num_kv_heads=8,
         head_dim=128, dtype="fp8"),                                                      # G = 8
    dict(num_seqs=5, prefix_len=500, suffix_min=1, suffix_max=9, num_q_heads=10, num_kv_heads=2,
         head_dim=128, dtype="fp8"),                                                      # G = 5
    dict(num_seqs=7, prefix_len=333, suffix_min=1, suffix_max=20, num_q_heads=8, num_kv_heads=8,
         head_dim=128, dtype="fp8"),                                                      # G = 1
]


@pytest.mark.parametrize("kernel", ["tcgen05", "mma_sync"])
@pytest.mark.parametrize("kw", SHARED, ids=[f"case{i}" for i in range(len(SHARED))])
def test_shared_prefix_parity(kw, kernel):
    """pa_decode_shared on fp8 pools, on the tcgen05 kernel (codes widened to f16
    in shared memory by converter warps) and on the mma.sync form: query heads
    per KV head 1, 4, 5 and 8, a span over two 1024-token chunks, three tiles
    of members; codes bit-exact, every output row within FP8_TOL of float64
    attention over the codes' values."""
    wl = wls.make_workload("prefix", **kw)
    values = wls.generate_values(wl, "cuda")
    pool, bm, setup_pairs = runtime.replay_setup(wl, values, "cuda")
    pool.set_option("shared_kernel", 1 if kernel == "mma_sync" else 0)
    step = runtime.prepare_step(wl, values, pool, bm, shared=True)
    step.run()
    torch.cuda.synchronize()
    assert step.sharing()
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert setup_pairs == st.setup_pairs
    assert_pools_equal(pool, st)
    ref = orp.attention(wl, values, st, threads=4)
    err = np.abs(step.out.double().cpu().numpy() - ref).max()
    assert err <= FP8_TOL, f"max-abs {err:.3g} > {FP8_TOL}"


@pytest.mark.parametrize("kernel", ["tcgen05", "mma_sync"])
def test_prefix_full_size_shared_parity(kernel):
    """The prefix workload (256 forks of a 4104-token prompt) on an fp8 pool
    through pa_decode_shared: the shared span read once per tile of members,
    on the tcgen05 kernel (codes widened to f16 in shared memory by converter
    warps) and on the mma.sync form (codes widened at fragment load); codes
    bit-exact, attention on sampled sequences."""
    wl = wls.make_workload("prefix", dtype="fp8")
    values = wls.generate_values(wl, "cuda")
    pool, bm, setup_pairs = runtime.replay_setup(wl, values, "cuda")
    pool.set_option("shared_kernel", 1 if kernel == "mma_sync" else 0)
    step = runtime.prepare_step(wl, values, pool, bm, shared=True)
    step.run()
    torch.cuda.synchronize()
    assert step.sharing()
    assert pool.get_error() == 0
    st = orp.replay(wl, values)
    assert setup_pairs == st.setup_pairs
    assert_pools_equal(pool, st)
    seqs = [0, 1, 100, wl.num_seqs - 1]
    ref = orp.attention(wl, values, st, seqs=seqs, threads=8)
    got = step.out.double().cpu().numpy()[np.asarray(seqs)]
    err = np.abs(got - ref).max()
    assert err <= FP8_TOL, f"max-abs {err:.3g} > {FP8_TOL}"
