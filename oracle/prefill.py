"""Paged prefill attention oracle (float64) — TEST INFRASTRUCTURE.

kgptalkie "Day 28: PagedAttention / vLLM" and the zenaique prefix-sharing
answer name the prefill step only through what a prefix-cache hit saves (a
hit means the cached span needs no prefill): a request's prompt tokens are processed
before it decodes, and their keys and values fill its blocks.  This build's
reading of one prefill chunk of a sequence (n new tokens, context length L
after they are appended):

* the chunk's keys and values are written first, at positions L-n .. L-1 of
  the sequence's block table (the append of ``kvcache.append_kv``);
* the query of chunk token i sits at position L-n+i and attends, through the
  same table, to every cached key at positions 0 .. L-n+i: the whole cached
  prefix, and the chunk causally up to itself.

So each chunk query is a decode query whose context ends at its own position,
and that is how it is computed here: one row per query token through the
float64 loops of ``attention.paged_decode`` (translation, two-pass softmax,
value mix), with the row's table the sequence's table and its length its
position + 1.
"""
import numpy as np

from .attention import paged_decode


def query_positions(cu_seqlens_q, context_lens):
    """(sequence of each query row, position of each query row)."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    L = np.asarray(context_lens, dtype=np.int64)
    n = np.diff(cu)
    if cu[0] != 0 or np.any(n < 0) or np.any(n > L):
        raise ValueError("cu_seqlens_q must start at 0, grow, and give chunks within the context")
    seq = np.repeat(np.arange(len(n)), n)
    pos = L[seq] - n[seq] + (np.arange(int(cu[-1])) - cu[seq])
    return seq, pos


def paged_prefill(q, k_pool, v_pool, block_tables, cu_seqlens_q, context_lens, scale,
                  num_kv_heads, threads: int = 1) -> np.ndarray:
    """Prefill attention of packed chunk queries q [T, Hq, D] (sequence s owns
    rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1) over paged pools
    ([num_blocks, Hkv, B, D], the storage kinds of ``paged_decode``).  Returns
    out [T, Hq, D] float64."""
    seq, pos = query_positions(cu_seqlens_q, context_lens)
    tables = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32)[seq])
    lens = (pos + 1).astype(np.int32)
    return paged_decode(q, k_pool, v_pool, tables, lens, scale, num_kv_heads, threads=threads)
