"""Decode attention oracle (float64) — TEST INFRASTRUCTURE.

Thin ctypes front end to the plain C loops in ``pa_oracle.c``:

* ``paged_decode``      — each sequence's query scores every cached key found
  through its block table in logical order (kgptalkie "Day 28: PagedAttention /
  vLLM", "The Block Table Is the Map", "Follow One Token Address", "Batching
  Becomes More Flexible"), softmax, then the value mix.
* ``contiguous_decode`` — the same maths on keys stored back to back, the
  "contiguous reference" of the verification recipe under "A Tiny Block-Table
  Example".

Pools and key/value arrays are numpy arrays in the oracle's own logical layout
``[num_blocks][Hkv][block_size][D]``, either float32 or the raw bits of
bfloat16 (uint16); the C loops widen every element exactly to float64, and all
arithmetic is float64.
"""
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        lp = ctypes.POINTER(ctypes.c_int64)
        i = ctypes.c_int
        vp = ctypes.c_void_p
        lib.oracle_paged_decode_range.argtypes = [i, i, i, i, i, i, dp, vp, vp, i, i, ip, i, ip,
                                                  ctypes.c_double, dp]
        lib.oracle_paged_decode_range.restype = i
        lib.oracle_contiguous_decode.argtypes = [i, i, i, i, dp, vp, vp, i, lp, ip,
                                                 ctypes.c_double, dp]
        lib.oracle_contiguous_decode.restype = i
        lib.oracle_translate.argtypes = [ctypes.c_int64, i, ip, i, lp]
        lib.oracle_translate.restype = i
        _LIB = lib
    return _LIB


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _kind(a) -> int:
    """0 for float32 storage, 1 for raw bfloat16 bits (uint16), 2 for float64
    (fp8 codes already turned into their values, see ``oracle.fp8``)."""
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float64:
        return 2
    raise TypeError("pool storage must be float32, uint16 bf16 bits or float64")


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 is the top half of an IEEE float32: widen the bits exactly."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def translate_c(pos: int, block_size: int, table) -> tuple:
    """The C loops' own translation routine, exposed so tests can pin it to the
    worked example ("Follow One Token Address")."""
    t = np.ascontiguousarray(table, dtype=np.int32)
    off = ctypes.c_int64(0)
    phys = _lib().oracle_translate(int(pos), int(block_size), _ptr(t, ctypes.c_int32),
                                   len(t), ctypes.byref(off))
    if phys < 0:
        raise ValueError("position outside the block table")
    return phys, off.value


def paged_decode(q, k_pool, v_pool, block_tables, context_lens, scale, num_kv_heads,
                 threads: int = 1) -> np.ndarray:
    """Paged decode attention in float64.

    q            [S, Hq, D]              any float dtype (upcast to float64)
    k_pool,v_pool[num_blocks, Hkv, B, D] float32, uint16 bfloat16 bits, or float64
    block_tables [S, max_blocks]         int32
    context_lens [S]                     int32 — tokens each query sees
    Returns out [S, Hq, D] float64.  ``threads`` splits the batch by sequence
    across host threads (the C routine releases the GIL through ctypes).
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k_pool = np.ascontiguousarray(k_pool)
    v_pool = np.ascontiguousarray(v_pool)
    kind = _kind(k_pool)
    if _kind(v_pool) != kind:
        raise TypeError("k_pool and v_pool storage differ")
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, Hq, D = q.shape
    nb, hkv, B, d2 = k_pool.shape
    if hkv != num_kv_heads or d2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("pool shape does not match the query")
    if tables.ndim != 2 or tables.shape[0] != S or lens.shape != (S,):
        raise ValueError("block_tables / context_lens shape")
    out = np.zeros((S, Hq, D), dtype=np.float64)
    lib = _lib()

    def run(lo, hi):
        return lib.oracle_paged_decode_range(
            lo, hi, Hq, hkv, D, B, _ptr(q, ctypes.c_double), k_pool.ctypes.data,
            v_pool.ctypes.data, kind, nb, _ptr(tables, ctypes.c_int32), tables.shape[1],
            _ptr(lens, ctypes.c_int32), float(scale), _ptr(out, ctypes.c_double))

    if threads <= 1 or S <= 1:
        rcs = [run(0, S)]
    else:
        edges = np.linspace(0, S, min(threads, S) + 1).astype(int)
        with ThreadPoolExecutor(max_workers=len(edges) - 1) as ex:
            rcs = list(ex.map(lambda ab: run(*ab), zip(edges[:-1], edges[1:])))
    for rc in rcs:
        if rc == -2:
            raise ValueError("block table entry outside the pool")
        if rc != 0:
            raise ValueError(f"oracle_paged_decode failed ({rc})")
    return out


def contiguous_decode(q, k_seqs, v_seqs, scale, num_kv_heads) -> np.ndarray:
    """Decode attention with each sequence's keys/values stored contiguously.

    k_seqs, v_seqs: lists of [L_s, Hkv, D] arrays (L_s may be 0), float32 or
    uint16 bfloat16 bits.
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    S, Hq, D = q.shape
    lens = np.array([k.shape[0] for k in k_seqs], dtype=np.int32)
    starts = np.zeros(S, dtype=np.int64)
    if S > 1:
        starts[1:] = np.cumsum(lens[:-1])
    store = np.asarray(k_seqs[0]).dtype if S else np.float32
    if lens.sum() > 0:
        kc = np.ascontiguousarray(np.concatenate([np.asarray(k, store) for k in k_seqs]))
        vc = np.ascontiguousarray(np.concatenate([np.asarray(v, store) for v in v_seqs]))
    else:
        kc = np.zeros((1, num_kv_heads, D), store)
        vc = np.zeros((1, num_kv_heads, D), store)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _lib().oracle_contiguous_decode(
        S, Hq, num_kv_heads, D, _ptr(q, ctypes.c_double), kc.ctypes.data, vc.ctypes.data,
        _kind(kc), _ptr(starts, ctypes.c_int64), _ptr(lens, ctypes.c_int32),
        float(scale), _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_contiguous_decode failed ({rc})")
    return out


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)
