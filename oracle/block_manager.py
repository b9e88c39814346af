"""Naive block-manager model — TEST INFRASTRUCTURE.

Plain Python lists and dicts for the host bookkeeping the pages describe:

* free pool, growth by one block at a block boundary — kgptalkie "Day 28",
  "Growth Needs Only Another Free Block" (9 tokens at block size 4 use 3
  blocks; tokens 10-12 need no allocation; the 13th needs a 4th block) and the
  "pool of free blocks" it maintains;
* per-block reference counts — zenaique "prefix sharing" answer and kgptalkie
  "Shared Blocks Must Not Be Changed in Place": a block is freed only when its
  last user leaves;
* copy-on-write — a write into a block that another request still points at
  allocates a fresh block, copies the old one, writes there and repoints only
  that entry of the writer's table (zenaique answer; kgptalkie "Shared Blocks
  Must Not Be Changed in Place"; zenaique "Most common mistake": the copy
  is limited to the single block where the requests diverge);
* parent-chained block hash and the hash -> physical block table — zenaique
  answer (each block's hash covers its own token ids and the hash of the
  block before it; a hit reuses the cached block and saves that span's
  prefill), its follow-ups on why the parent's hash is chained in and on what
  else must enter the cache key (here: a per-request salt), and kgptalkie
  "Prefix Reuse Also Needs Compatible Computation" (only full blocks are kept
  for reuse, so only full blocks are hashed).

Readings where the pages are silent (each listed in the design notes):
  - the free pool is a FIFO seeded with a caller-given order; freed blocks go
    to its tail, in logical table order;
  - block hash h_i = FNV-1a-64 over (h_{i-1} as 8 little-endian bytes,
    salt as 8 LE bytes, the block's token ids as 4 LE bytes each), h_{-1} = 0;
  - a hit also checks the stored token ids and parent block (collision guard);
  - a full block is registered when it becomes full; if an identical chain is
    already registered the first registration stays;
  - a block leaves the hash table when its reference count reaches zero,
    unless retention is on.  Retention (the zenaique follow-up on how eviction
    interacts with the reference count is left unanswered; kgptalkie leaves
    what to keep for reuse to each system's policy): a registered
    block whose count reaches zero stays registered and evictable, in release
    order; a finished request releases its blocks last one first; a new block
    comes from the free pool while it has one, else the least recently
    released evictable block is evicted (it leaves the hash table); an
    admission hit on an evictable block takes it back;
  - a write into a block with reference count 1 happens in place.
"""
from collections import deque

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


class BlockManagerError(Exception):
    pass


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    """FNV-1a, 64-bit: for each byte, xor it in, then multiply by the prime."""
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent_hash: int, salt: int, tokens) -> int:
    data = (parent_hash & MASK64).to_bytes(8, "little") + (salt & MASK64).to_bytes(8, "little")
    for t in tokens:
        data += (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
    return fnv1a64(data)


class NaiveBlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None, retain=False):
        if num_blocks <= 0 or block_size <= 0:
            raise BlockManagerError("bad pool size")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise BlockManagerError("free order must be a permutation of the pool")
        self.free = deque(order)
        self.refcount = [0] * num_blocks
        self.cache = {}          # hash -> (block, parent block, tokens tuple)
        self.block_key = {}      # registered block -> hash
        self.requests = {}       # id -> dict(table, tokens, hashes, salt)
        self.next_id = 0
        self.retain = bool(retain)
        self.evictable = []      # registered blocks nobody holds, least recently released first

    # -- helpers ---------------------------------------------------------
    def _take_free(self) -> int:
        if self.free:
            return self.free.popleft()
        if self.evictable:                      # evict the least recently released cached block
            blk = self.evictable.pop(0)
            del self.cache[self.block_key.pop(blk)]
            return blk
        raise BlockManagerError("no free block")

    def _release(self, blk: int):
        if self.refcount[blk] <= 0:
            raise BlockManagerError("refcount underflow")
        self.refcount[blk] -= 1
        if self.refcount[blk] == 0:
            if blk in self.block_key:
                if self.retain:
                    self.evictable.append(blk)
                    return
                del self.cache[self.block_key.pop(blk)]
            self.free.append(blk)

    def _req(self, rid: int) -> dict:
        if rid not in self.requests:
            raise BlockManagerError("unknown request")
        return self.requests[rid]

    # -- operations ------------------------------------------------------
    def add_request(self, prompt_tokens, salt: int = 0):
        """Admit a request: reuse cached full prefix blocks while they hit.

        Returns (request id, number of prompt tokens served from the cache).
        The caller appends the remaining prompt tokens with append_slot.
        """
        B = self.block_size
        req = dict(table=[], tokens=[], hashes=[], salt=int(salt))
        parent_hash, parent_blk = 0, -1
        for i in range(len(prompt_tokens) // B):
            toks = tuple(int(t) for t in prompt_tokens[i * B:(i + 1) * B])
            h = block_hash(parent_hash, salt, toks)
            entry = self.cache.get(h)
            if entry is None or entry[1] != parent_blk or entry[2] != toks:
                break
            blk = entry[0]
            if self.refcount[blk] == 0:
                self.evictable.remove(blk)      # in use again
            self.refcount[blk] += 1
            req["table"].append(blk)
            req["tokens"].extend(toks)
            req["hashes"].append(h)
            parent_hash, parent_blk = h, blk
        rid = self.next_id
        self.next_id += 1
        self.requests[rid] = req
        return rid, len(req["tokens"])

    def fork(self, parent_id: int) -> int:
        """A child request that shares every block of its parent."""
        p = self._req(parent_id)
        for blk in p["table"]:
            self.refcount[blk] += 1
        rid = self.next_id
        self.next_id += 1
        self.requests[rid] = dict(table=list(p["table"]), tokens=list(p["tokens"]),
                                  hashes=list(p["hashes"]), salt=p["salt"])
        return rid

    def append_slot(self, rid: int, token: int):
        """Reserve the slot of the request's next token.

        Returns (slot, cow_src, cow_dst); cow_src = cow_dst = -1 when no copy is
        needed.  On error the state is unchanged.
        """
        req = self._req(rid)
        B = self.block_size
        pos = len(req["tokens"])
        logical, offset = divmod(pos, B)
        cow = (-1, -1)
        if offset == 0:
            blk = self._take_free()
            self.refcount[blk] = 1
            req["table"].append(blk)
        else:
            blk = req["table"][logical]
            if self.refcount[blk] > 1:
                fresh = self._take_free()
                self.refcount[blk] -= 1
                self.refcount[fresh] = 1
                req["table"][logical] = fresh
                cow = (blk, fresh)
                blk = fresh
        req["tokens"].append(int(token))
        if offset == B - 1:
            toks = tuple(req["tokens"][logical * B:(logical + 1) * B])
            parent_hash = req["hashes"][-1] if req["hashes"] else 0
            h = block_hash(parent_hash, req["salt"], toks)
            req["hashes"].append(h)
            if h not in self.cache:
                parent_blk = req["table"][logical - 1] if logical > 0 else -1
                self.cache[h] = (blk, parent_blk, toks)
                self.block_key[blk] = h
        return blk * B + offset, cow[0], cow[1]

    def free_request(self, rid: int):
        req = self._req(rid)
        for blk in (reversed(req["table"]) if self.retain else req["table"]):
            self._release(blk)
        del self.requests[rid]

    def set_retention(self, on: bool):
        if not on:                               # retained blocks rejoin the free pool
            for blk in self.evictable:
                del self.cache[self.block_key.pop(blk)]
                self.free.append(blk)
            self.evictable = []
        self.retain = bool(on)

    # -- queries ---------------------------------------------------------
    def block_table(self, rid: int) -> list:
        return list(self._req(rid)["table"])

    def seq_len(self, rid: int) -> int:
        return len(self._req(rid)["tokens"])

    def num_free(self) -> int:
        return len(self.free)

    def is_cached(self, blk: int) -> bool:
        return blk in self.block_key
