"""KV-cache data movement oracle — TEST INFRASTRUCTURE.

Bit-level reference for the two data-movement steps around decode attention.
Pools are numpy arrays of raw element bits (uint16 for bf16, uint32 for
float32) in the oracle's logical layout ``[num_blocks][Hkv][block_size][D]``,
so comparisons are exact.

* ``translate``    — kgptalkie "Day 28", "Follow One Token Address": logical
  block and offset are ``divmod(position, block_size)``; the block table maps
  the logical block to a physical one.
* ``append_kv``    — zenaique "prefix sharing" answer (a new token "is written
  there") and kgptalkie "Growth Needs Only Another Free Block": each new
  token's keys and values land in its (physical block, offset) slot.  Slots
  are encoded ``physical_block * block_size + offset``; a negative slot means
  "no write".
* ``copy_blocks``  — kgptalkie "Shared Blocks Must Not Be Changed in Place":
  copy-on-write makes a private copy of the whole shared block (every slot,
  keys and values) before the diverging write.
"""
import numpy as np


def translate(position: int, block_size: int, block_table) -> tuple:
    """(physical block, offset) of a token position."""
    logical_block, offset = divmod(int(position), int(block_size))
    return int(block_table[logical_block]), offset


def slot_of(position: int, block_size: int, block_table) -> int:
    phys, off = translate(position, block_size, block_table)
    return phys * block_size + off


def append_kv(k_pool, v_pool, k_new, v_new, slot_mapping):
    """Write token t's rows k_new[t] / v_new[t] ([Hkv, D] each) into its slot.

    For every t with slot_mapping[t] >= 0:
        block, offset = divmod(slot, block_size)
        K[block, :, offset, :] = k_new[t];  V[block, :, offset, :] = v_new[t]
    (one numpy fancy-indexed assignment per pool).  Pools are modified in place
    and returned.  Raises on a slot outside the pool.
    """
    nb, hkv, B, D = k_pool.shape
    slots = np.asarray(slot_mapping, dtype=np.int64).reshape(-1)
    keep = slots >= 0
    blk, off = np.divmod(slots[keep], B)
    if blk.size and blk.max() >= nb:
        raise ValueError("slot outside the pool")
    k_pool[blk, :, off, :] = np.asarray(k_new)[keep]
    v_pool[blk, :, off, :] = np.asarray(v_new)[keep]
    return k_pool, v_pool


def copy_blocks(k_pool, v_pool, pairs):
    """For each (src, dst) pair copy block src's keys and values to block dst.

    Pairs are applied in order; the pairs a block manager emits for
    copy-on-write never overlap (a destination is always a fresh block).
    """
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        k_pool[dst] = k_pool[src]
        v_pool[dst] = v_pool[src]
    return k_pool, v_pool
