"""ctypes binding of libpagedattn.so — argument marshalling only.

Every function of ``include/pa.h`` is exposed under its own name with its C
signature.  All computation happens in the library's CUDA kernels (or, for
the block manager, its C++ host code); nothing here has a fallback: if the
library is missing, importing this module raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpagedattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libpagedattn.so not built ({LIB_PATH} missing); run "
        "`python -m paged_kv_cache_253_gb300.build` or __graft_entry__.build()")

lib = ctypes.CDLL(LIB_PATH)

c_int, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
c_i32p = ctypes.POINTER(ctypes.c_int32)
c_i64p = ctypes.POINTER(ctypes.c_int64)
c_u8p = ctypes.POINTER(ctypes.c_uint8)
c_intp = ctypes.POINTER(c_int)

PA_F32, PA_BF16, PA_FP8E4M3 = 0, 1, 2
PA_OPT_PARTITION_CAP, PA_OPT_SHARED_KERNEL, PA_OPT_PREFILL_KERNEL = 0, 1, 2

ERRORS = {
    0: "PA_OK", -1: "PA_ERR_INVALID_ARG", -2: "PA_ERR_DTYPE", -3: "PA_ERR_CUDA",
    -4: "PA_ERR_NO_FREE_BLOCK", -5: "PA_ERR_BAD_BLOCK_ID", -6: "PA_ERR_BAD_SLOT",
    -7: "PA_ERR_REFCOUNT", -8: "PA_ERR_UNKNOWN_REQUEST", -9: "PA_ERR_OUT_OF_MEMORY",
    -10: "PA_ERR_UNSUPPORTED", -11: "PA_ERR_OVERLAP", -12: "PA_ERR_BAD_LENGTH",
}
globals().update({v: k for k, v in ERRORS.items()})

# name -> (restype, argtypes): one entry per declaration of pa.h
SIGNATURES = {
    "pa_pool_create": (c_int, [c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(c_void_p)]),
    "pa_pool_destroy": (c_int, [c_void_p]),
    "pa_pool_kv_ptrs": (c_int, [c_void_p, ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p)]),
    "pa_pool_export": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "pa_pool_import": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "pa_pool_info": (c_int, [c_void_p, c_intp, c_intp, c_intp, c_intp, c_intp]),
    "pa_pool_set_kv_scales": (c_int, [c_void_p, c_float, c_float]),
    "pa_pool_kv_scales": (c_int, [c_void_p, ctypes.POINTER(c_float), ctypes.POINTER(c_float)]),
    "pa_pool_set_option": (c_int, [c_void_p, c_int, c_int]),
    "pa_pool_get_option": (c_int, [c_void_p, c_int, c_intp]),
    "pa_append_kv": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "pa_copy_blocks": (c_int, [c_void_p, c_void_p, c_int, c_void_p]),
    "pa_decode": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_int, c_void_p, c_float,
                          c_void_p, c_int, c_void_p]),
    "pa_decode_reserve": (c_int, [c_void_p, c_int, c_int]),
    "pa_append_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                 c_void_p, c_int, c_void_p, c_float, c_void_p, c_int, c_void_p]),
    "pa_decode_shared": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_int, c_void_p,
                                 c_float, c_void_p, c_int, c_i32p, c_i32p, c_i32p, c_int,
                                 c_void_p]),
    "pa_decode_noalloc": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_int, c_void_p,
                                  c_float, c_void_p, c_int, c_void_p]),
    "pa_prefill": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_int, c_int, c_void_p,
                           c_int, c_void_p, c_float, c_void_p, c_int, c_void_p]),
    "pa_get_error": (c_int, [c_void_p, c_void_p]),
    "pa_error_string": (ctypes.c_char_p, [c_int]),
    "pa_launch_count": (ctypes.c_uint64, []),
    "pa_bm_create": (c_int, [c_int, c_int, c_i32p, ctypes.POINTER(c_void_p)]),
    "pa_bm_destroy": (c_int, [c_void_p]),
    "pa_bm_add_request": (c_int, [c_void_p, c_i32p, c_int, ctypes.c_uint64, c_intp, c_intp]),
    "pa_bm_fork": (c_int, [c_void_p, c_int, c_intp]),
    "pa_bm_append_slot": (c_int, [c_void_p, c_int, ctypes.c_int32, c_i64p, c_i64p, c_i64p]),
    "pa_bm_append_slots": (c_int, [c_void_p, c_int, c_i32p, c_i32p, c_i64p, c_i64p, c_intp,
                                   c_intp]),
    "pa_bm_free_request": (c_int, [c_void_p, c_int]),
    "pa_bm_block_table": (c_int, [c_void_p, c_int, c_i32p, c_int, c_intp]),
    "pa_bm_batch_tables": (c_int, [c_void_p, c_int, c_i32p, c_int, c_i32p, c_i32p]),
    "pa_bm_batch_width": (c_int, [c_void_p, c_int, c_i32p, c_intp]),
    "pa_bm_seq_len": (c_int, [c_void_p, c_int]),
    "pa_bm_refcount": (c_int, [c_void_p, c_int]),
    "pa_bm_num_free": (c_int, [c_void_p]),
    "pa_bm_free_list": (c_int, [c_void_p, c_i32p, c_int, c_intp]),
    "pa_bm_is_cached": (c_int, [c_void_p, c_int]),
    "pa_bm_set_retention": (c_int, [c_void_p, c_int]),
    "pa_bm_num_evictable": (c_int, [c_void_p]),
    "pa_bm_evictable_list": (c_int, [c_void_p, c_i32p, c_int, c_intp]),
    "pa_bm_prefix_groups": (c_int, [c_void_p, c_int, c_i32p, c_i32p, c_i32p, c_i32p, c_intp]),
    "pa_bm_fnv1a64": (ctypes.c_uint64, [c_u8p, c_size_t]),
}

for _name, (_res, _args) in SIGNATURES.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn


class PagedAttnError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = lib.pa_error_string(code).decode()
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({msg})" if what else msg)


def check(code, what=""):
    if code != 0:
        raise PagedAttnError(code, what)
    return code
