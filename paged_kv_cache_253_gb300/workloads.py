"""Seeded synthetic workloads for the paged decode step.

This module is shared by the tests, the benchmark and the oracle harness, and
therefore holds none of the method's arithmetic: no address translation, no
block allocation, no attention.  It only draws the random inputs that
describe a workload —

* the pool geometry (block size, heads, head width, dtype, number of blocks),
* the order in which the pool's blocks sit in the free list (a seeded
  permutation, which is what makes every block table a scattered draw of
  physical blocks),
* a setup script of host events: admit a request with its prompt token ids
  (``add``), fork a request so the child shares all of its blocks
  (``fork``), and append token ids to a request (``extend``),
* the decode step: which requests are in the batch, in which order, and the
  token each one appends,

and, separately, the floating-point values (queries, and keys/values of every
token that the script appends) from a seeded torch generator.

Each side (the CUDA library with its C++ block manager, or the oracle with its
naive model) replays the script through its own bookkeeping.

Workloads (sizes from the pages' problem statement for this build):
  tiny     block_size 4, 16 blocks, 3 requests of 9/3/5 cached tokens,
           2 q heads / 2 KV heads, head_dim 8, float32
  decode   64 sequences, lengths U[128, 2048], block_size 16, 32 q / 8 KV
           heads, head_dim 128, bf16, pool 1.25x the blocks needed
  prefix   256 requests forked from one 4104-token prompt (256 full blocks and
           a partly filled one, all shared), unique suffixes U[64, 512]
  long     8 sequences, lengths U[32768, 131072], pool 1.1x demand
  mixed    512 sequences, lognormal lengths (median 1024, sigma 1, clipped to
           [16, 16384]), 64 q / 8 KV heads; 30 % of the requests are forks
           of one of 4 prompts of U[512, 2048] tokens that diverge in the
           timed step
  prefill  16 sequences with cached prefixes U[0, 4096] and a chunk of
           U[128, 512] new tokens each (chunked prefill: the step appends the
           chunk and runs its queries), 32 q / 8 KV heads, head_dim 128, bf16
"""
from dataclasses import dataclass, field
import math

import numpy as np

VOCAB = 32000

WORKLOAD_NAMES = ("tiny", "decode", "prefix", "long", "mixed", "prefill")


@dataclass
class Workload:
    name: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f32", "bf16" or "fp8" (e4m3 pool, bf16 inputs)
    num_blocks: int
    free_order: np.ndarray          # int32 permutation of range(num_blocks)
    events: list                    # ("add", rid, tokens, salt) | ("fork", rid, parent)
                                    # | ("extend", rid, tokens)
    batch: np.ndarray               # int32 request ids of the decode batch, in order
    step_tokens: np.ndarray         # int32 token id each batch entry appends
    scale: float
    seed: int
    shared_groups: list = field(default_factory=list)  # [rid, ...] lists forked together
    description: str = ""
    kv_scales: tuple = (1.0, 1.0)   # fp8 pool: (k_scale, v_scale), float32 values
    # prefill step: batch entry i appends chunk_lens[i] tokens (step_tokens holds
    # them all, entry after entry) and runs their queries; None: one decode token
    chunk_lens: np.ndarray = None

    @property
    def num_seqs(self) -> int:
        return int(len(self.batch))

    @property
    def num_step_tokens(self) -> int:
        """Tokens the timed step appends (and queries it runs)."""
        return int(self.chunk_lens.sum()) if self.chunk_lens is not None else self.num_seqs

    @property
    def num_history_tokens(self) -> int:
        return int(sum(len(e[2]) for e in self.events if e[0] == "extend"))

    @property
    def elem_bytes(self) -> int:
        """Bytes of one pool element."""
        return {"f32": 4, "bf16": 2, "fp8": 1}[self.dtype]

    @property
    def input_dtype(self) -> str:
        """Element type of q and of the appended keys and values."""
        return "f32" if self.dtype == "f32" else "bf16"


def _tokens(rng, n):
    return rng.integers(0, VOCAB, size=int(n), dtype=np.int64).astype(np.int32)


def _blocks_for(n_tokens, block_size):
    # a count of tokens rounded up to whole blocks: sizing the pool only
    return -(-int(n_tokens) // int(block_size))


def _independent(name, rng, lengths, B, hq, hkv, d, dtype, pool_factor, seed, desc):
    """Requests without sharing: admit, append the cached history, one step token."""
    events = []
    for rid, L in enumerate(lengths):
        toks = _tokens(rng, L)
        events.append(("add", rid, toks, 0))
        events.append(("extend", rid, toks))
    need = sum(_blocks_for(L + 1, B) for L in lengths)
    nb = max(int(math.ceil(need * pool_factor)), need)
    return Workload(name=name, block_size=B, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                    dtype=dtype, num_blocks=nb,
                    free_order=rng.permutation(nb).astype(np.int32), events=events,
                    batch=np.arange(len(lengths), dtype=np.int32),
                    step_tokens=_tokens(rng, len(lengths)), scale=1.0 / math.sqrt(d),
                    seed=seed, description=desc)


# Scales of an fp8 pool: N(0,1) keys and values then span about +-7 of e4m3's
# +-448 (no saturation in practice); two unequal values that are not powers
# of two, so that the division before rounding is not exact and a K/V mix-up
# shows.
FP8_KV_SCALES = (0.0173, 0.0141)


def make_workload(name: str, seed: int = None, **kw) -> Workload:
    """Build one of the named workloads.

    Keyword overrides shrink a workload for parity tests (``num_seqs``,
    ``min_len``/``max_len``, ``prefix_len``, ``suffix_min``/``suffix_max``,
    ``num_prefixes``, ``share_frac``, ``num_q_heads``, ``num_kv_heads``,
    ``head_dim``, ``block_size``, ``dtype``, ``pool_factor``, ``lengths``,
    ``kv_scales`` for dtype "fp8").
    """
    wl = _make(name, seed, **kw)
    if wl.dtype == "fp8":
        ks, vs = kw.get("kv_scales", FP8_KV_SCALES)
        wl.kv_scales = (float(np.float32(ks)), float(np.float32(vs)))
        wl.description += ", fp8 e4m3 pool"
    elif wl.dtype not in ("f32", "bf16"):
        raise ValueError(f"unknown dtype {wl.dtype!r}")
    return wl


def _make(name, seed, **kw):
    if name not in WORKLOAD_NAMES:
        raise ValueError(f"unknown workload {name!r}")
    if seed is None:
        seed = 253 + WORKLOAD_NAMES.index(name)
    rng = np.random.default_rng(seed)

    if name == "tiny":
        B = kw.get("block_size", 4)
        lengths = list(kw.get("lengths", [9, 3, 5]))
        nb = kw.get("num_blocks", 16)
        hq, hkv, d = kw.get("num_q_heads", 2), kw.get("num_kv_heads", 2), kw.get("head_dim", 8)
        events = []
        for rid, L in enumerate(lengths):
            toks = _tokens(rng, L)
            events.append(("add", rid, toks, 0))
            events.append(("extend", rid, toks))
        return Workload(name=name, block_size=B, num_q_heads=hq, num_kv_heads=hkv,
                        head_dim=d, dtype=kw.get("dtype", "f32"), num_blocks=nb,
                        free_order=rng.permutation(nb).astype(np.int32), events=events,
                        batch=np.arange(len(lengths), dtype=np.int32),
                        step_tokens=_tokens(rng, len(lengths)),
                        scale=1.0 / math.sqrt(d), seed=seed,
                        description="3 requests, block_size 4, fp32")

    B = kw.get("block_size", 16)
    d = kw.get("head_dim", 128)
    dtype = kw.get("dtype", "bf16")

    if name in ("decode", "long"):
        if name == "decode":
            S, lo, hi, hq, hkv, pf = 64, 128, 2048, 32, 8, 1.25
        else:
            S, lo, hi, hq, hkv, pf = 8, 32768, 131072, 32, 8, 1.1
        S = kw.get("num_seqs", S)
        lo, hi = kw.get("min_len", lo), kw.get("max_len", hi)
        hq, hkv = kw.get("num_q_heads", hq), kw.get("num_kv_heads", hkv)
        pf = kw.get("pool_factor", pf)
        lengths = kw.get("lengths")
        if lengths is None:
            lengths = rng.integers(lo, hi + 1, size=S).tolist()
        return _independent(name, rng, [int(x) for x in lengths], B, hq, hkv, d, dtype, pf,
                            seed, f"{len(lengths)} sequences, lengths U[{lo},{hi}]")

    if name == "prefix":
        S = kw.get("num_seqs", 256)
        plen = kw.get("prefix_len", 4104)
        smin, smax = kw.get("suffix_min", 64), kw.get("suffix_max", 512)
        hq, hkv = kw.get("num_q_heads", 32), kw.get("num_kv_heads", 8)
        prefix = _tokens(rng, plen)
        events = [("add", 0, prefix, 0), ("extend", 0, prefix)]
        for rid in range(1, S):
            events.append(("fork", rid, 0))
        suffix_lens = rng.integers(smin, smax + 1, size=S)
        for rid in range(S):
            events.append(("extend", rid, _tokens(rng, suffix_lens[rid])))
        need = _blocks_for(plen, B) + sum(
            _blocks_for(plen + int(sl) + 1, B) - plen // B for sl in suffix_lens)
        nb = int(math.ceil(need * kw.get("pool_factor", 1.25)))
        return Workload(name=name, block_size=B, num_q_heads=hq, num_kv_heads=hkv,
                        head_dim=d, dtype=dtype, num_blocks=nb,
                        free_order=rng.permutation(nb).astype(np.int32), events=events,
                        batch=np.arange(S, dtype=np.int32), step_tokens=_tokens(rng, S),
                        scale=1.0 / math.sqrt(d), seed=seed,
                        shared_groups=[list(range(S))],
                        description=f"{S} requests forked from a {plen}-token prompt")

    if name == "prefill":
        S = kw.get("num_seqs", 16)
        hq, hkv = kw.get("num_q_heads", 32), kw.get("num_kv_heads", 8)
        plo, phi = kw.get("min_len", 0), kw.get("max_len", 4096)
        clo, chi = kw.get("chunk_min", 128), kw.get("chunk_max", 512)
        prefix = kw.get("lengths")
        if prefix is None:
            prefix = rng.integers(plo, phi + 1, size=S).tolist()
        chunks = kw.get("chunks")
        if chunks is None:
            chunks = rng.integers(clo, chi + 1, size=len(prefix)).tolist()
        events = []
        for rid, L in enumerate(prefix):
            toks = _tokens(rng, L)
            events.append(("add", rid, toks, 0))
            events.append(("extend", rid, toks))
        chunk_lens = np.asarray(chunks, dtype=np.int32)
        need = sum(_blocks_for(int(L) + int(c), B) for L, c in zip(prefix, chunks))
        nb = int(math.ceil(need * kw.get("pool_factor", 1.1))) + 1
        return Workload(name=name, block_size=B, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                        dtype=dtype, num_blocks=nb,
                        free_order=rng.permutation(nb).astype(np.int32), events=events,
                        batch=np.arange(len(prefix), dtype=np.int32),
                        step_tokens=_tokens(rng, int(chunk_lens.sum())),
                        scale=1.0 / math.sqrt(d), seed=seed, chunk_lens=chunk_lens,
                        description=f"{len(prefix)} sequences, cached prefixes U[{plo},{phi}], "
                                    f"chunks U[{clo},{chi}]")

    # mixed
    S = kw.get("num_seqs", 512)
    hq, hkv = kw.get("num_q_heads", 64), kw.get("num_kv_heads", 8)
    median, sigma = kw.get("median", 1024), kw.get("sigma", 1.0)
    lo, hi = kw.get("min_len", 16), kw.get("max_len", 16384)
    n_pref = kw.get("num_prefixes", 4)
    pmin, pmax = kw.get("prefix_min", 512), kw.get("prefix_max", 2048)
    frac = kw.get("share_frac", 0.30)
    n_share = int(round(frac * S))
    lengths = np.clip(np.round(rng.lognormal(math.log(median), sigma, size=S)), lo, hi)
    lengths = lengths.astype(np.int64)
    prefix_lens = rng.integers(pmin, pmax + 1, size=n_pref)
    order = rng.permutation(S)          # batch position -> request slot
    share_of = -np.ones(S, dtype=np.int64)
    share_of[order[:n_share]] = rng.integers(0, n_pref, size=n_share)
    events, groups = [], []
    rid = 0
    rid_of_slot = np.zeros(S, dtype=np.int64)
    for g in range(n_pref):
        members = [i for i in range(S) if share_of[i] == g]
        if not members:
            continue
        toks = _tokens(rng, prefix_lens[g])
        root = rid
        events.append(("add", root, toks, 0))
        events.append(("extend", root, toks))
        rid_of_slot[members[0]] = root
        rid += 1
        grp = [root]
        for m in members[1:]:
            events.append(("fork", rid, root))
            rid_of_slot[m] = rid
            grp.append(rid)
            rid += 1
        groups.append(grp)
    for i in range(S):
        if share_of[i] >= 0:
            continue
        toks = _tokens(rng, lengths[i])
        events.append(("add", rid, toks, 0))
        events.append(("extend", rid, toks))
        rid_of_slot[i] = rid
        rid += 1
    batch = rid_of_slot[rng.permutation(S)].astype(np.int32)
    need = sum(_blocks_for(int(lengths[i]) + 1, B) for i in range(S) if share_of[i] < 0)
    need += sum(_blocks_for(int(prefix_lens[g]), B) + len([i for i in range(S) if share_of[i] == g])
                for g in range(n_pref))
    nb = int(math.ceil(need * kw.get("pool_factor", 1.25)))
    return Workload(name=name, block_size=B, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                    dtype=dtype, num_blocks=nb, free_order=rng.permutation(nb).astype(np.int32),
                    events=events, batch=batch, step_tokens=_tokens(rng, S),
                    scale=1.0 / math.sqrt(d), seed=seed, shared_groups=groups,
                    description=f"{S} sequences, lognormal lengths, {n_share} forks of "
                                f"{n_pref} prompts diverging this step")


def generate_values(wl: Workload, device="cpu", seed: int = None):
    """Seeded float inputs: q [T,Hq,D], hist_k/hist_v [N_hist,Hkv,D] (the keys and
    values of every token the setup script appends, in script order) and
    new_k/new_v [T,Hkv,D] (the tokens the step appends: one per batch entry for
    a decode step, T = S; each entry's chunk, entry after entry, for a prefill
    step, T = sum of chunk_lens).

    Values are N(0,1) draws in float32 from a torch generator on ``device``,
    rounded once to the workload's input dtype (bf16 for an fp8 pool); both
    sides read those same values.
    """
    import torch
    if seed is None:
        seed = wl.seed
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    dt = torch.float32 if wl.input_dtype == "f32" else torch.bfloat16
    S, hq, hkv, d = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    n_hist = wl.num_history_tokens

    def draw(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dt)

    T = wl.num_step_tokens          # one query / new token per decode entry, a chunk per prefill entry
    return dict(q=draw(T, hq, d), hist_k=draw(n_hist, hkv, d), hist_v=draw(n_hist, hkv, d),
                new_k=draw(T, hkv, d), new_v=draw(T, hkv, d))
