"""Replay a workload script through the oracle — TEST INFRASTRUCTURE.

Runs the host events of a workload (admit, fork, append) through the naive
block manager, applying every copy-on-write copy and every key/value write to
the oracle's own bit-level pools in the order the events happen, then runs the
decode step (each batch entry appends its token, then attends over all of its
cached tokens, its new one included) and the float64 attention.

An fp8 workload's pools hold e4m3 codes: each appended bf16 row is quantized
with the pool's K or V scale when it is written, and the attention reads the
codes' values times the scales (the e4m3 format and its rounding are in
fp8.py).

The only thing shared with the GPU side is the workload description and the
seeded values; the bookkeeping, the data movement and the attention are all
the oracle's own.
"""
import numpy as np

from . import fp8
from .attention import paged_decode
from .block_manager import NaiveBlockManager
from .kvcache import append_kv, copy_blocks
from .prefill import paged_prefill


def values_to_numpy(t):
    """A torch tensor of seeded values as numpy: float32 stays float32,
    bfloat16 becomes its raw bits (uint16)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy().astype(np.float32, copy=False)


def _bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _stored(wl, t, which):
    """Rows as the pool stores them: the input bits, or for an fp8 pool the
    e4m3 codes of the bf16 values under the K (which=0) or V (which=1) scale."""
    x = values_to_numpy(t)
    if wl.dtype != "fp8":
        return x
    out = np.empty(x.shape, dtype=np.uint8)
    step = max(1, (1 << 22) // max(1, int(np.prod(x.shape[1:]))))     # bounded temporaries
    for lo in range(0, x.shape[0], step):
        out[lo:lo + step] = fp8.quantize(_bf16_bits_to_f32(x[lo:lo + step]), wl.kv_scales[which])
    return out


class OracleState:
    """Result of a replay: pools after the step, the step's device inputs as the
    oracle derived them, and (optionally) the attention output."""

    def __init__(self):
        self.k_pool = self.v_pool = None
        self.setup_pairs = []
        self.step_pairs = []
        self.step_slots = None
        self.block_tables = None
        self.context_lens = None
        self.cu_seqlens_q = None       # prefill step: query rows of each batch entry
        self.bm = None


def replay(wl, values, *, run_step=True):
    """Replay ``wl``'s setup script (and its decode-step appends if run_step)."""
    st = OracleState()
    bm = NaiveBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    store = {"f32": np.float32, "bf16": np.uint16, "fp8": np.uint8}[wl.dtype]
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    K = np.zeros(shape, store)
    V = np.zeros(shape, store)
    hk = _stored(wl, values["hist_k"], 0)
    hv = _stored(wl, values["hist_v"], 1)
    row = 0
    pend_slots, pend_rows, pend_set = [], [], set()

    def flush():
        if pend_slots:
            rows = np.asarray(pend_rows, dtype=np.int64)
            append_kv(K, V, hk[rows], hv[rows], np.asarray(pend_slots, dtype=np.int64))
            pend_slots.clear()
            pend_rows.clear()
            pend_set.clear()

    for ev in wl.events:
        kind = ev[0]
        if kind == "add":
            rid, _ = bm.add_request(ev[2], ev[3])
            assert rid == ev[1]
        elif kind == "fork":
            rid = bm.fork(ev[2])
            assert rid == ev[1]
        elif kind == "extend":
            for tok in np.asarray(ev[2]).tolist():
                slot, src, dst = bm.append_slot(ev[1], tok)
                if src >= 0:
                    flush()                     # the copy must see every earlier write
                    copy_blocks(K, V, [(src, dst)])
                    st.setup_pairs.append((src, dst))
                if slot in pend_set:            # a slot written twice: keep the order
                    flush()
                pend_slots.append(slot)
                pend_set.add(slot)
                pend_rows.append(row)
                row += 1
        else:
            raise ValueError(kind)
    flush()

    if run_step:
        nk = _stored(wl, values["new_k"], 0)
        nv = _stored(wl, values["new_v"], 1)
        slots = []
        # decode: one token per batch entry; prefill: each entry's chunk, in order
        per_entry = wl.chunk_lens if wl.chunk_lens is not None else np.ones(wl.num_seqs, np.int64)
        r = 0
        for i, rid in enumerate(wl.batch.tolist()):
            for _ in range(int(per_entry[i])):
                slot, src, dst = bm.append_slot(rid, int(wl.step_tokens[r]))
                if src >= 0:
                    copy_blocks(K, V, [(src, dst)])
                    st.step_pairs.append((src, dst))
                append_kv(K, V, nk[r:r + 1], nv[r:r + 1], [slot])
                slots.append(slot)
                r += 1
        st.step_slots = np.asarray(slots, dtype=np.int64)
        st.cu_seqlens_q = np.concatenate([[0], np.cumsum(per_entry)]).astype(np.int32)

    S = wl.num_seqs
    tables = [bm.block_table(r) for r in wl.batch.tolist()]
    width = max(1, max(len(t) for t in tables))
    bt = np.full((S, width), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    st.block_tables = bt
    st.context_lens = np.asarray([bm.seq_len(r) for r in wl.batch.tolist()], dtype=np.int32)
    st.k_pool, st.v_pool, st.bm = K, V, bm
    return st


def _pools_for(wl, st, bt):
    """The pools the attention reads and the tables into them: the stored bits
    as they are, or for an fp8 pool the values its codes stand for (code value
    times the K or V scale), of the blocks these tables reach only (renumbered
    so that only those are widened to float64)."""
    kp, vp = st.k_pool, st.v_pool
    if wl.dtype != "fp8":
        return kp, vp, bt
    used = np.unique(bt[bt >= 0])
    renum = np.full(kp.shape[0], -1, dtype=np.int32)
    renum[used] = np.arange(len(used), dtype=np.int32)
    bt = np.where(bt >= 0, renum[np.maximum(bt, 0)], -1).astype(np.int32)
    return fp8.dequantize(kp[used], wl.kv_scales[0]), fp8.dequantize(vp[used], wl.kv_scales[1]), bt


def attention(wl, values, st, seqs=None, threads=1):
    """float64 decode attention for all batch entries (or the listed ones)."""
    q = values_to_numpy(values["q"])
    if q.dtype == np.uint16:
        q = _bf16_bits_to_f32(q)
    bt, lens = st.block_tables, st.context_lens
    if seqs is not None:
        seqs = np.asarray(seqs, dtype=np.int64)
        q, bt, lens = q[seqs], bt[seqs], lens[seqs]
    kp, vp, bt = _pools_for(wl, st, bt)
    return paged_decode(q, kp, vp, bt, lens, wl.scale, wl.num_kv_heads, threads=threads)


def prefill_attention(wl, values, st, seqs=None, threads=1):
    """float64 prefill attention of the step's chunk queries, for all batch
    entries or the listed ones (rows of those entries, entry after entry)."""
    q = values_to_numpy(values["q"])
    if q.dtype == np.uint16:
        q = _bf16_bits_to_f32(q)
    cu, bt, lens = st.cu_seqlens_q, st.block_tables, st.context_lens
    if seqs is not None:
        seqs = np.asarray(seqs, dtype=np.int64)
        rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]) if len(seqs) else \
            np.zeros(0, np.int64)
        n = cu[seqs + 1] - cu[seqs]
        q, bt, lens = q[rows], bt[seqs], lens[seqs]
        cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    kp, vp, bt = _pools_for(wl, st, bt)
    return paged_prefill(q, kp, vp, bt, cu, lens, wl.scale, wl.num_kv_heads, threads=threads)
