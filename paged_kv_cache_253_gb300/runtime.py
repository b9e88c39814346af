"""Drive a workload through the library: host block manager + GPU kernels.

``replay_setup`` runs a workload's setup script (admit / fork / append)
through the C++ block manager and issues the pool writes it implies on the
GPU: copy-on-write copies through ``pa_copy_blocks`` and key/value writes
through ``pa_append_kv``, batched, but each copy issued after every write it
depends on and before every write into its destination.

``prepare_step`` then reserves the decode step's slots (one new token per
batch entry, with any copy-on-write pairs) and uploads the step's inputs.
``DecodeStep.run`` issues the step: copies, append, decode — three library
calls on the current stream.
"""
from dataclasses import dataclass
import time

import numpy as np
import torch

from .api import BlockManager, KVPool


def _dtype(wl):
    return torch.float32 if wl.input_dtype == "f32" else torch.bfloat16


class _Writer:
    """Batches pool writes while keeping the order that the script implies."""

    def __init__(self, pool, hist_k, hist_v, device):
        self.pool, self.hk, self.hv, self.device = pool, hist_k, hist_v, device
        self.rows_lo = None          # pending appends: history rows [lo, hi) ...
        self.rows_hi = None
        self.slots = []              # ... and their slots
        self.slot_set = set()
        self.pairs = []              # pending copies
        self.pair_blocks = set()
        self.setup_pairs = []

    def flush_appends(self):
        if self.slots:
            s = torch.as_tensor(np.concatenate(self.slots), device=self.device)
            self.pool.append_kv(self.hk[self.rows_lo:self.rows_hi],
                                self.hv[self.rows_lo:self.rows_hi], s)
            self.slots, self.slot_set = [], set()
            self.rows_lo = self.rows_hi = None

    def flush_copies(self):
        if self.pairs:
            p = torch.as_tensor(np.asarray(self.pairs, dtype=np.int64), device=self.device)
            self.pool.copy_blocks(p)
            self.pairs, self.pair_blocks = [], set()

    def copy(self, src, dst):
        self.flush_appends()                          # the copy reads every earlier write
        if src in self.pair_blocks or dst in self.pair_blocks:
            self.flush_copies()
        self.pairs.append((src, dst))
        self.pair_blocks.update((src, dst))
        self.setup_pairs.append((src, dst))

    def append(self, row_lo, slots):
        self.flush_copies()                           # writes land after the copies
        if self.rows_hi is not None and (row_lo != self.rows_hi or
                                         any(int(x) in self.slot_set for x in slots)):
            self.flush_appends()
        if self.rows_lo is None:
            self.rows_lo = row_lo
        self.rows_hi = row_lo + len(slots)
        self.slots.append(np.asarray(slots, dtype=np.int64))
        self.slot_set.update(int(x) for x in slots)


def replay_setup(wl, values, device=None):
    """Returns (pool, bm, setup copy pairs) with the pool holding the history."""
    device = torch.device(device) if device is not None else torch.device("cuda")
    pool = KVPool(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, wl.dtype, device)
    if wl.dtype == "fp8":
        pool.set_kv_scales(*wl.kv_scales)
    bm = BlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    hk = values["hist_k"].to(device).contiguous()
    hv = values["hist_v"].to(device).contiguous()
    w = _Writer(pool, hk, hv, pool.device)
    row = 0
    for ev in wl.events:
        if ev[0] == "add":
            rid, _ = bm.add_request(ev[2], ev[3])
            assert rid == ev[1], "request ids follow admission order"
        elif ev[0] == "fork":
            rid = bm.fork(ev[2])
            assert rid == ev[1]
        elif ev[0] == "extend":
            toks = np.asarray(ev[2], dtype=np.int32)
            if len(toks) == 0:
                continue
            # only a request's first new token can land in a shared block
            slot, src, dst = bm.append_slot(ev[1], int(toks[0]))
            if src >= 0:
                w.copy(src, dst)
            w.append(row, [slot])
            if len(toks) > 1:
                slots, pairs = bm.append_slots(np.full(len(toks) - 1, ev[1], np.int32), toks[1:])
                if len(pairs):
                    raise RuntimeError("copy-on-write after a request's first new token")
                w.append(row + 1, slots)
            row += len(toks)
    w.flush_copies()
    w.flush_appends()
    return pool, bm, w.setup_pairs


@dataclass
class DecodeStep:
    """Device inputs of one decode step and the calls that run it."""
    pool: KVPool
    q: torch.Tensor
    new_k: torch.Tensor
    new_v: torch.Tensor
    slots: torch.Tensor            # int64 [S]
    pairs: torch.Tensor            # int64 [P, 2]
    block_tables: torch.Tensor     # int32 [S, W]
    context_lens: torch.Tensor     # int32 [S], after the append
    scale: float
    out: torch.Tensor
    groups: tuple = None           # (offsets, seqs, shared_blocks): decode with shared reads
    fused: bool = True             # append inside the decode kernel when there is no sharing
    host_ms: float = 0.0           # host block-manager time of the step (slots, tables, groups)

    @property
    def num_pairs(self):
        return int(self.pairs.shape[0])

    def decode(self):
        if self.groups is not None and len(self.groups[2]):
            return self.pool.decode_shared(self.q, self.block_tables, self.context_lens,
                                           self.scale, self.groups, out=self.out)
        return self.pool.decode(self.q, self.block_tables, self.context_lens, self.scale,
                                out=self.out)

    def sharing(self):
        return self.groups is not None and len(self.groups[2]) > 0

    def run(self):
        if self.num_pairs:
            self.pool.copy_blocks(self.pairs)
        if self.fused and not self.sharing():
            self.pool.append_decode(self.new_k, self.new_v, self.slots, self.q, self.block_tables,
                                    self.context_lens, self.scale, out=self.out)
            return self.out
        self.pool.append_kv(self.new_k, self.new_v, self.slots)
        self.decode()
        return self.out


SHARED_MIN_FRACTION = 0.5


def shared_fraction(groups, lens, block_size):
    """Fraction of a step's logical KV reads that fall in shared spans."""
    offs, seqs, nsh = groups
    shared = sum((int(offs[g + 1]) - int(offs[g])) * int(nsh[g]) * block_size
                 for g in range(len(nsh)))
    return shared / max(1, int(np.asarray(lens).sum()))


def prepare_step(wl, values, pool, bm, out_dtype=torch.float32, shared="auto", fused=True):
    """Reserve the step's slots in the block manager and upload its inputs.

    shared=True decodes through pa_decode_shared whenever the block manager
    finds batch entries that share leading blocks; "auto" does so only when the
    shared spans are at least SHARED_MIN_FRACTION of the step's logical KV
    reads (below that, L2 already absorbs the repeated reads and the plain
    kernel's higher occupancy wins, as measured on the mixed workload)."""
    dev = pool.device
    t0 = time.perf_counter()
    slots, pairs = bm.append_slots(wl.batch, wl.step_tokens)
    tables, lens = bm.batch_tables(wl.batch)
    groups = bm.prefix_groups(wl.batch) if shared else None
    if shared == "auto" and groups is not None and \
            shared_fraction(groups, lens, wl.block_size) < SHARED_MIN_FRACTION:
        groups = None
    host_ms = (time.perf_counter() - t0) * 1e3
    S = wl.num_seqs
    return DecodeStep(
        pool=pool,
        q=values["q"].to(dev).contiguous(),
        new_k=values["new_k"].to(dev).contiguous(),
        new_v=values["new_v"].to(dev).contiguous(),
        slots=torch.as_tensor(slots, device=dev),
        pairs=torch.as_tensor(pairs.reshape(-1, 2), device=dev),
        block_tables=torch.as_tensor(tables, device=dev),
        context_lens=torch.as_tensor(lens, device=dev),
        scale=wl.scale,
        out=torch.empty((S, wl.num_q_heads, wl.head_dim), dtype=out_dtype, device=dev),
        groups=groups, fused=fused, host_ms=host_ms)


@dataclass
class PrefillStep:
    """Device inputs of one chunked-prefill step and the calls that run it."""
    pool: KVPool
    q: torch.Tensor                # [T, Hq, D]
    new_k: torch.Tensor            # [T, Hkv, D]
    new_v: torch.Tensor
    slots: torch.Tensor            # int64 [T]
    pairs: torch.Tensor            # int64 [P, 2]
    cu_seqlens_q: torch.Tensor     # int32 [S + 1]
    max_q_len: int
    block_tables: torch.Tensor     # int32 [S, W]
    context_lens: torch.Tensor     # int32 [S], after the chunk's append
    scale: float
    out: torch.Tensor              # [T, Hq, D]
    host_ms: float = 0.0           # host block-manager time of the step (slots, tables)

    @property
    def num_pairs(self):
        return int(self.pairs.shape[0])

    def sharing(self):
        return False

    def attend(self):
        return self.pool.prefill(self.q, self.cu_seqlens_q, self.block_tables, self.context_lens,
                                 self.scale, max_q_len=self.max_q_len, out=self.out)

    def run(self):
        if self.num_pairs:
            self.pool.copy_blocks(self.pairs)
        self.pool.append_kv(self.new_k, self.new_v, self.slots)
        self.attend()
        return self.out


def prepare_prefill(wl, values, pool, bm, out_dtype=torch.float32):
    """Reserve the slots of every chunk token (entry after entry, each entry's
    tokens in order) and upload the step's inputs."""
    dev = pool.device
    t0 = time.perf_counter()
    reqs = np.repeat(np.asarray(wl.batch, dtype=np.int32), wl.chunk_lens)
    slots, pairs = bm.append_slots(reqs, wl.step_tokens)
    tables, lens = bm.batch_tables(wl.batch)
    host_ms = (time.perf_counter() - t0) * 1e3
    cu = np.zeros(len(wl.chunk_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(wl.chunk_lens)
    T = int(cu[-1])
    return PrefillStep(
        pool=pool, q=values["q"].to(dev).contiguous(),
        new_k=values["new_k"].to(dev).contiguous(), new_v=values["new_v"].to(dev).contiguous(),
        slots=torch.as_tensor(slots, device=dev),
        pairs=torch.as_tensor(pairs.reshape(-1, 2), device=dev),
        cu_seqlens_q=torch.as_tensor(cu, device=dev),
        max_q_len=int(np.max(wl.chunk_lens)) if len(wl.chunk_lens) else 0,
        block_tables=torch.as_tensor(tables, device=dev),
        context_lens=torch.as_tensor(lens, device=dev), scale=wl.scale,
        out=torch.empty((T, wl.num_q_heads, wl.head_dim), dtype=out_dtype, device=dev),
        host_ms=host_ms)
