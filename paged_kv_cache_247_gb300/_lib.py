"""ctypes declarations of ``libpagedkv.so`` (the C ABI in include/pagedkv.h).

Argument marshalling only: every step of the device path runs in the
library's kernels.  Loading fails loudly when the library has not been built.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

c_int, c_int64, c_size_t, c_float, c_void_p = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                               ctypes.c_float, ctypes.c_void_p)
P_i32 = ctypes.POINTER(ctypes.c_int32)
P_i64 = ctypes.POINTER(ctypes.c_int64)
P_int = ctypes.POINTER(ctypes.c_int)
P_u32 = ctypes.POINTER(ctypes.c_uint32)

STATUS = {
    0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
    3: "PKV_ERR_WORKSPACE_TOO_SMALL", 4: "PKV_ERR_OUT_OF_BLOCKS", 5: "PKV_ERR_CUDA",
    6: "PKV_ERR_UNKNOWN_SEQ", 7: "PKV_ERR_SEQ_EXISTS", 8: "PKV_ERR_TABLE_TOO_SMALL",
}
PKV_F16, PKV_BF16 = 0, 1
DEV_BAD_BLOCK_ID, DEV_BAD_CONTEXT_LEN, DEV_BAD_SLOT, DEV_WAIT_TIMEOUT = 1, 2, 4, 8


class AllocStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in (
        "num_blocks", "free_blocks", "used_blocks", "shared_blocks", "num_seqs",
        "logical_tokens", "filled_slots", "cow_copies")]


# name -> (restype, argtypes)
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [c_int]),
    "pkv_last_cuda_error": (c_int, []),
    "pkv_version": (c_int, []),
    "pkv_paged_attn_decode": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int,
        c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_int, c_void_p, c_size_t,
        c_void_p]),
    "pkv_paged_attn_decode_append": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
        c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_int, c_void_p,
        c_size_t, c_void_p]),
    "pkv_paged_attn_decode_noalloc": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int,
        c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_int, c_void_p]),
    "pkv_contiguous_attn_decode": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
        c_float, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "pkv_paged_attn_prefill": (c_int, [
        c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int,
        c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "pkv_decode_partition_size": (c_int, [c_int, c_int, c_int, c_int, c_int]),
    "pkv_set_decode_path": (c_int, [c_int]),
    "pkv_get_decode_path": (c_int, []),
    "pkv_decode_uses_tensor_cores": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "pkv_decode_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "pkv_contiguous_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "pkv_kv_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                              c_int, c_int, c_int, c_int, c_void_p]),
    "pkv_block_copy": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_size_t, c_void_p]),
    "pkv_device_status": (c_int, [P_u32, c_int, c_void_p]),
    "pkv_debug_wait_timeout": (c_int, [c_void_p]),
    "pkv_alloc_create": (c_int, [c_int, c_int, ctypes.POINTER(c_void_p)]),
    "pkv_alloc_destroy": (None, [c_void_p]),
    "pkv_alloc_add_seq": (c_int, [c_void_p, c_int64, c_int]),
    "pkv_alloc_fork": (c_int, [c_void_p, c_int64, c_int64]),
    "pkv_alloc_append_slot": (c_int, [c_void_p, c_int64, P_i64, P_i64, P_i64]),
    # array arguments are passed as addresses (numpy's .ctypes.data), which
    # costs half as much per call as building typed pointers
    "pkv_alloc_append_slots": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, P_int]),
    "pkv_alloc_free_seq": (c_int, [c_void_p, c_int64]),
    "pkv_alloc_block_table": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int]),
    "pkv_alloc_seq_slots": (c_int, [c_void_p, c_int64, c_int, c_int, c_void_p]),
    "pkv_alloc_seq_info": (c_int, [c_void_p, c_int64, P_int, P_int]),
    "pkv_alloc_refcount": (c_int, [c_void_p, c_int, P_int]),
    "pkv_alloc_stats": (c_int, [c_void_p, ctypes.POINTER(AllocStats)]),
}

_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        name = STATUS.get(status, str(status))
        extra = ""
        if status == 5 and _lib is not None:
            extra = f" (cudaError {_lib.pkv_last_cuda_error()})"
        super().__init__(f"{what}: {name}{extra}")


def load():
    """Load the library once and attach the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with paged_kv_cache_247_gb300.build.build_library() "
            "(there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status, what):
    if status != 0:
        raise PagedKVError(status, what)
