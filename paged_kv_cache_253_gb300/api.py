"""Python front end of the C ABI: torch tensors in, raw pointers out.

PyTorch provides device memory and the current CUDA stream; every step of the
path runs in libpagedattn's kernels.  Argument checks here only guard the
pointer marshalling (device, dtype, contiguity, shape).
"""
import ctypes

import numpy as np
import torch

from . import _lib as L

# pool element type -> (torch type of k/v/q inputs, torch type of the stored elements)
_TORCH = {L.PA_F32: (torch.float32, torch.float32), L.PA_BF16: (torch.bfloat16, torch.bfloat16),
          L.PA_FP8E4M3: (torch.bfloat16, torch.uint8)}
_CODE = {torch.float32: L.PA_F32, torch.bfloat16: L.PA_BF16, "f32": L.PA_F32,
         "bf16": L.PA_BF16, "fp8": L.PA_FP8E4M3, "fp8e4m3": L.PA_FP8E4M3}


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t, dtype, name, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device != device:
        raise ValueError(f"{name} must live on {device}, got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _i32p(a):
    return a.ctypes.data_as(L.c_i32p)


class KVPool:
    """A pool of fixed-size physical KV blocks on one GPU (one layer).

    K is [num_blocks, kv_heads, block_size, head_dim]; V is stored transposed
    per tile, [num_blocks, kv_heads, head_dim, block_size].  dtype "fp8" keeps
    one e4m3 code per element (stored as uint8; a code stands for its value
    times the pool's K or V scale) and takes bf16 k, v and q.
    """

    def __init__(self, num_blocks, block_size, kv_heads, head_dim, dtype="bf16", device=None):
        dev = torch.device("cuda") if device is None else torch.device(device)
        if dev.type != "cuda":
            raise ValueError("KVPool lives on a CUDA device")
        self.device = dev if dev.index is not None else torch.device("cuda", torch.cuda.current_device())
        self.dtype_code = _CODE[dtype]
        self.dtype, self.storage_dtype = _TORCH[self.dtype_code]
        self.fp8 = self.dtype_code == L.PA_FP8E4M3
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.kv_heads, self.head_dim = int(kv_heads), int(head_dim)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            L.check(L.pa_pool_create(self.num_blocks, self.block_size, self.kv_heads,
                                     self.head_dim, self.dtype_code, ctypes.byref(h)),
                    "pa_pool_create")
        self.handle = h

    def set_kv_scales(self, k_scale, v_scale):
        """Scales of an fp8 pool (set them before the first append)."""
        L.check(L.pa_pool_set_kv_scales(self.handle, float(k_scale), float(v_scale)),
                "pa_pool_set_kv_scales")

    def kv_scales(self):
        k, v = ctypes.c_float(), ctypes.c_float()
        L.check(L.pa_pool_kv_scales(self.handle, ctypes.byref(k), ctypes.byref(v)),
                "pa_pool_kv_scales")
        return k.value, v.value

    OPTIONS = {"partition_cap": L.PA_OPT_PARTITION_CAP, "shared_kernel": L.PA_OPT_SHARED_KERNEL,
               "prefill_kernel": L.PA_OPT_PREFILL_KERNEL}

    def set_option(self, name, value):
        """Kernel-choice option of this pool (pa_pool_set_option): partition_cap
        (tokens; 0 none, -1 automatic), shared_kernel / prefill_kernel (0
        tcgen05 where eligible, 1 mma.sync)."""
        L.check(L.pa_pool_set_option(self.handle, self.OPTIONS[name], int(value)),
                "pa_pool_set_option")

    def get_option(self, name):
        v = ctypes.c_int()
        L.check(L.pa_pool_get_option(self.handle, self.OPTIONS[name], ctypes.byref(v)),
                "pa_pool_get_option")
        return v.value

    def close(self):
        if getattr(self, "handle", None):
            L.pa_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- data movement ---------------------------------------------------
    def append_kv(self, k, v, slot_mapping):
        T = int(slot_mapping.shape[0])
        shape = (T, self.kv_heads, self.head_dim)
        if tuple(k.shape) != shape or tuple(v.shape) != shape:
            raise ValueError(f"k/v must be {shape}")
        L.check(L.pa_append_kv(self.handle, _dev(k, self.dtype, "k", self.device),
                               _dev(v, self.dtype, "v", self.device),
                               _dev(slot_mapping, torch.int64, "slot_mapping", self.device), T,
                               _stream()), "pa_append_kv")

    def copy_blocks(self, pairs):
        P = int(pairs.shape[0]) if pairs.numel() else 0
        if P and tuple(pairs.shape) != (P, 2):
            raise ValueError("pairs must be [P, 2]")
        ptr = _dev(pairs, torch.int64, "pairs", self.device) if P else None
        L.check(L.pa_copy_blocks(self.handle, ptr, P, _stream()), "pa_copy_blocks")

    def decode(self, q, block_tables, context_lens, scale, out=None, out_dtype=torch.float32):
        S, hq, d = q.shape
        if d != self.head_dim:
            raise ValueError("q head_dim does not match the pool")
        if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
            raise ValueError("block_tables [S, max_blocks] / context_lens [S]")
        if out is None:
            out = torch.empty((S, hq, d), dtype=out_dtype, device=self.device)
        if tuple(out.shape) != (S, hq, d):
            raise ValueError("out must be [S, Hq, D]")
        L.check(L.pa_decode(self.handle, _dev(q, self.dtype, "q", self.device), S, hq,
                            _dev(block_tables, torch.int32, "block_tables", self.device),
                            int(block_tables.shape[1]),
                            _dev(context_lens, torch.int32, "context_lens", self.device),
                            float(scale), _dev(out, out.dtype, "out", self.device),
                            _CODE[out.dtype], _stream()), "pa_decode")
        return out

    def append_decode(self, k, v, slot_mapping, q, block_tables, context_lens, scale, out=None,
                      out_dtype=torch.float32):
        """Write each sequence's new token (k[s], v[s] at slot_mapping[s]), then decode."""
        S, hq, d = q.shape
        shape = (S, self.kv_heads, self.head_dim)
        if tuple(k.shape) != shape or tuple(v.shape) != shape or tuple(slot_mapping.shape) != (S,):
            raise ValueError(f"k/v must be {shape}, slot_mapping [S]")
        if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
            raise ValueError("block_tables [S, max_blocks] / context_lens [S]")
        if out is None:
            out = torch.empty((S, hq, d), dtype=out_dtype, device=self.device)
        L.check(L.pa_append_decode(self.handle, _dev(k, self.dtype, "k", self.device),
                                   _dev(v, self.dtype, "v", self.device),
                                   _dev(slot_mapping, torch.int64, "slot_mapping", self.device),
                                   _dev(q, self.dtype, "q", self.device), S, hq,
                                   _dev(block_tables, torch.int32, "block_tables", self.device),
                                   int(block_tables.shape[1]),
                                   _dev(context_lens, torch.int32, "context_lens", self.device),
                                   float(scale), _dev(out, out.dtype, "out", self.device),
                                   _CODE[out.dtype], _stream()), "pa_append_decode")
        return out

    def decode_shared(self, q, block_tables, context_lens, scale, groups, out=None,
                      out_dtype=torch.float32):
        """Decode with shared leading blocks read once per group.

        groups = (offsets, seqs, shared_blocks) host int32 arrays, as returned by
        BlockManager.prefix_groups.
        """
        offs, seqs, nsh = (np.ascontiguousarray(a, dtype=np.int32) for a in groups)
        S, hq, d = q.shape
        if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
            raise ValueError("block_tables [S, max_blocks] / context_lens [S]")
        if out is None:
            out = torch.empty((S, hq, d), dtype=out_dtype, device=self.device)
        ng = len(nsh)
        if len(offs) != ng + 1:
            raise ValueError("group offsets must have num_groups + 1 entries")
        L.check(L.pa_decode_shared(self.handle, _dev(q, self.dtype, "q", self.device), S, hq,
                                   _dev(block_tables, torch.int32, "block_tables", self.device),
                                   int(block_tables.shape[1]),
                                   _dev(context_lens, torch.int32, "context_lens", self.device),
                                   float(scale), _dev(out, out.dtype, "out", self.device),
                                   _CODE[out.dtype], _i32p(offs), _i32p(seqs) if len(seqs) else None,
                                   _i32p(nsh) if ng else None, ng, _stream()),
                "pa_decode_shared")
        return out

    def prefill(self, q, cu_seqlens_q, block_tables, context_lens, scale, max_q_len=None,
                out=None, out_dtype=torch.float32):
        """Chunked prefill: the packed chunk queries q [T, Hq, D] (sequence s owns
        rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1) attend to the cached prefix
        and causally to their chunk.  The chunk's keys and values must already
        be appended.  max_q_len (longest chunk) is read from cu_seqlens_q when
        not given (one device-to-host copy)."""
        T, hq, d = q.shape
        S = int(cu_seqlens_q.shape[0]) - 1
        if d != self.head_dim or S < 0:
            raise ValueError("q head_dim / cu_seqlens_q [S+1]")
        if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
            raise ValueError("block_tables [S, max_blocks] / context_lens [S]")
        if max_q_len is None:
            max_q_len = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if S else 0
        if out is None:
            out = torch.empty((T, hq, d), dtype=out_dtype, device=self.device)
        if tuple(out.shape) != (T, hq, d):
            raise ValueError("out must be [T, Hq, D]")
        L.check(L.pa_prefill(self.handle, _dev(q, self.dtype, "q", self.device), T, hq,
                             _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q", self.device), S,
                             int(max_q_len),
                             _dev(block_tables, torch.int32, "block_tables", self.device),
                             int(block_tables.shape[1]),
                             _dev(context_lens, torch.int32, "context_lens", self.device),
                             float(scale), _dev(out, out.dtype, "out", self.device),
                             _CODE[out.dtype], _stream()), "pa_prefill")
        return out

    def reserve(self, max_seqs, max_q_heads):
        L.check(L.pa_decode_reserve(self.handle, int(max_seqs), int(max_q_heads)),
                "pa_decode_reserve")

    def get_error(self):
        """Synchronise the current stream; return the recorded error code (0 = none)."""
        return L.pa_get_error(self.handle, _stream())

    def check_error(self):
        code = self.get_error()
        if code:
            raise L.PagedAttnError(code, "device")

    # -- snapshots ---------------------------------------------------------
    def export(self):
        """Copies of (K, V) as device tensors in the pool's own layout."""
        k = torch.empty((self.num_blocks, self.kv_heads, self.block_size, self.head_dim),
                        dtype=self.storage_dtype, device=self.device)
        v = torch.empty((self.num_blocks, self.kv_heads, self.head_dim, self.block_size),
                        dtype=self.storage_dtype, device=self.device)
        L.check(L.pa_pool_export(self.handle, ctypes.c_void_p(k.data_ptr()),
                                 ctypes.c_void_p(v.data_ptr()), _stream()), "pa_pool_export")
        return k, v

    def import_(self, k, v):
        L.check(L.pa_pool_import(self.handle, _dev(k, self.storage_dtype, "k", self.device),
                                 _dev(v, self.storage_dtype, "v", self.device), _stream()),
                "pa_pool_import")


class BlockManager:
    """Host free pool, reference counts, copy-on-write and prefix hash (C++)."""

    def __init__(self, num_blocks, block_size, free_order=None):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            order = _i32p(self._order)
        L.check(L.pa_bm_create(self.num_blocks, self.block_size, order, ctypes.byref(h)),
                "pa_bm_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            L.pa_bm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_request(self, tokens, salt=0):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        rid, cached = ctypes.c_int(), ctypes.c_int()
        L.check(L.pa_bm_add_request(self.handle, _i32p(t), len(t), ctypes.c_uint64(salt),
                                    ctypes.byref(rid), ctypes.byref(cached)), "pa_bm_add_request")
        return rid.value, cached.value

    def fork(self, parent):
        c = ctypes.c_int()
        L.check(L.pa_bm_fork(self.handle, int(parent), ctypes.byref(c)), "pa_bm_fork")
        return c.value

    def append_slot(self, req, token):
        slot, s, d = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        L.check(L.pa_bm_append_slot(self.handle, int(req), int(token), ctypes.byref(slot),
                                    ctypes.byref(s), ctypes.byref(d)), "pa_bm_append_slot")
        return slot.value, s.value, d.value

    def append_slots(self, reqs, tokens):
        """Batched appends: returns (slots int64 [n], pairs int64 [P, 2])."""
        r = np.ascontiguousarray(reqs, dtype=np.int32)
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = len(r)
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        npairs, done = ctypes.c_int(), ctypes.c_int()
        L.check(L.pa_bm_append_slots(self.handle, n, _i32p(r), _i32p(t),
                                     slots.ctypes.data_as(L.c_i64p),
                                     pairs.ctypes.data_as(L.c_i64p), ctypes.byref(npairs),
                                     ctypes.byref(done)), "pa_bm_append_slots")
        return slots, pairs[:npairs.value].copy()

    def free_request(self, req):
        L.check(L.pa_bm_free_request(self.handle, int(req)), "pa_bm_free_request")

    def block_table(self, req):
        n = ctypes.c_int()
        L.check(L.pa_bm_block_table(self.handle, int(req), None, 0, ctypes.byref(n)),
                "pa_bm_block_table")
        out = np.empty(max(n.value, 1), dtype=np.int32)
        L.check(L.pa_bm_block_table(self.handle, int(req), _i32p(out), n.value, ctypes.byref(n)),
                "pa_bm_block_table")
        return out[:n.value].tolist()

    def batch_tables(self, reqs, width=None):
        r = np.ascontiguousarray(reqs, dtype=np.int32)
        if width is None:
            w = ctypes.c_int()
            L.check(L.pa_bm_batch_width(self.handle, len(r), _i32p(r), ctypes.byref(w)),
                    "pa_bm_batch_width")
            width = max(1, w.value)
        tables = np.empty((len(r), width), dtype=np.int32)
        lens = np.empty(len(r), dtype=np.int32)
        L.check(L.pa_bm_batch_tables(self.handle, len(r), _i32p(r), int(width), _i32p(tables),
                                     _i32p(lens)), "pa_bm_batch_tables")
        return tables, lens

    def seq_len(self, req):
        return L.pa_bm_seq_len(self.handle, int(req))

    def refcount(self, block):
        return L.pa_bm_refcount(self.handle, int(block))

    def num_free(self):
        return L.pa_bm_num_free(self.handle)

    def free_list(self):
        n = ctypes.c_int()
        out = np.empty(self.num_blocks, dtype=np.int32)
        L.check(L.pa_bm_free_list(self.handle, _i32p(out), self.num_blocks, ctypes.byref(n)),
                "pa_bm_free_list")
        return out[:n.value].tolist()

    def prefix_groups(self, reqs):
        """(offsets, seqs, shared_blocks) of the batch's sharing groups."""
        r = np.ascontiguousarray(reqs, dtype=np.int32)
        n = len(r)
        offs = np.zeros(n + 1, dtype=np.int32)
        seqs = np.zeros(max(n, 1), dtype=np.int32)
        nsh = np.zeros(max(n, 1), dtype=np.int32)
        ng = ctypes.c_int()
        L.check(L.pa_bm_prefix_groups(self.handle, n, _i32p(r), _i32p(offs), _i32p(seqs),
                                      _i32p(nsh), ctypes.byref(ng)), "pa_bm_prefix_groups")
        g = ng.value
        return offs[:g + 1].copy(), seqs[:offs[g]].copy(), nsh[:g].copy()

    def is_cached(self, block):
        return L.pa_bm_is_cached(self.handle, int(block)) == 1

    def set_retention(self, on):
        L.check(L.pa_bm_set_retention(self.handle, 1 if on else 0), "pa_bm_set_retention")

    def num_evictable(self):
        return L.pa_bm_num_evictable(self.handle)

    def evictable_list(self):
        n = ctypes.c_int()
        out = np.empty(self.num_blocks, dtype=np.int32)
        L.check(L.pa_bm_evictable_list(self.handle, _i32p(out), self.num_blocks, ctypes.byref(n)),
                "pa_bm_evictable_list")
        return out[:n.value].tolist()


def fnv1a64(data: bytes) -> int:
    buf = (ctypes.c_uint8 * max(len(data), 1)).from_buffer_copy(data or b"\0")
    return int(L.pa_bm_fnv1a64(buf, len(data)))


def launch_count() -> int:
    return int(L.pa_launch_count())
