"""ctypes declarations of libspec.so (include/spec.h). Loading fails loudly if the library is
missing: there is no CPU fallback anywhere in this package."""

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspec.so")

SPEC_OK, SPEC_ERR_INVALID, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA = 0, 1, 2, 3
SPEC_BF16, SPEC_F32, SPEC_Q4A32 = 0, 1, 2
SPEC_COMMIT_SNAPSHOT, SPEC_COMMIT_REPLAY, SPEC_COMMIT_INDEX = 0, 1, 2
REQ_OK, REQ_NONFINITE, REQ_BAD_K, REQ_KV_OVERFLOW, REQ_NO_LOGITS, REQ_BAD_TOKEN, \
    REQ_BAD_FILTER = range(7)

# Exported symbols declared in include/spec.h (checked by the CPU test that loads the library).
EXPORTS = ("spec_workspace_bytes", "spec_status_str", "spec_lmhead_verify",
           "spec_verify_accept_greedy", "spec_draft_argmax",
           "spec_accept", "spec_accept_exact", "spec_accept_filtered", "spec_adapt_width",
           "spec_adapt_width_mirror",
           "spec_draft_argmax_rows", "spec_accept_rows",
           "spec_commit_rollback",
           "spec_batched_supported", "spec_host_alias", "spec_copy_from_host",
           "spec_lmhead_verify_noalloc", "spec_noalloc_scratch_bytes",
           "spec_noalloc_error_word", "spec_test_verify_stalled",
           "spec_width_graph_create", "spec_graph_capture_begin", "spec_graph_capture_end",
           "spec_graph_instantiate", "spec_graph_launch", "spec_graph_destroy")

# numpy views of the device structs (for reading results copied to the host)
ROWSTATS_DTYPE = np.dtype([("max", "<f4"), ("log_norm", "<f4"), ("gap", "<f4"),
                           ("argmax", "<i4")])
ACCEPT_OUT_DTYPE = np.dtype([("status", "<i4"), ("n_accept", "<i4"), ("n_emit", "<i4"),
                             ("eos_hit", "<i4"), ("tokens", "<i4", (8,)),
                             ("sample_kind", "<i4"), ("sample_row", "<i4"),
                             ("reserved", "<i4", (2,))])
WIDTH_STATE_DTYPE = np.dtype([("rate", "<f4", (8,)), ("seen", "<u4"), ("cycles", "<u4"),
                              ("k", "<i4"), ("t_last", "<u4"), ("fit", "<f4", (4,))])
COUNTERS_DTYPE = np.dtype([("cycles", "<u8"), ("drafted", "<u8"), ("accepted", "<u8"),
                           ("emitted", "<u8"), ("eos", "<u8"), ("errors", "<u8"),
                           ("depth", "<u8", (8,))])
assert ROWSTATS_DTYPE.itemsize == 16 and ACCEPT_OUT_DTYPE.itemsize == 64
assert COUNTERS_DTYPE.itemsize == 112


class spec_state_desc(ctypes.Structure):
    _fields_ = [
        ("kv", ctypes.c_void_p),
        ("kv_request_stride", ctypes.c_int64),
        ("kv_layers", ctypes.c_int32),
        ("kv_capacity", ctypes.c_int64),
        ("kv_row_bytes", ctypes.c_int64),
        ("kv_len", ctypes.c_void_p),
        ("rec_layers", ctypes.c_int32),
        ("rec_heads", ctypes.c_int32),
        ("rec_dk", ctypes.c_int32),
        ("rec_dv", ctypes.c_int32),
        ("rec_live", ctypes.c_void_p),
        ("rec_slots", ctypes.c_void_p),
        ("conv_rows", ctypes.c_int32),
        ("conv_width", ctypes.c_int32),
        ("conv_live", ctypes.c_void_p),
        ("conv_slots", ctypes.c_void_p),
        ("n_slots", ctypes.c_int32),
        ("step_a", ctypes.c_void_p),
        ("step_b", ctypes.c_void_p),
        ("step_c", ctypes.c_void_p),
        ("conv_in", ctypes.c_void_p),
        ("live_slot", ctypes.c_void_p),
    ]


_lib = None


def lib():
    """The loaded libspec.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libspec.so not found at {LIB_PATH}; build it with "
                "`python -m mtp_speculative_decoding_spec_gb300.build` (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.spec_workspace_bytes.argtypes = [i64, i32]
        L.spec_workspace_bytes.restype = sz
        L.spec_status_str.argtypes = [i32]
        L.spec_status_str.restype = ctypes.c_char_p
        L.spec_batched_supported.argtypes = []
        L.spec_batched_supported.restype = i32
        L.spec_host_alias.argtypes = [vp, ctypes.POINTER(ctypes.c_void_p)]
        L.spec_host_alias.restype = i32
        L.spec_copy_from_host.argtypes = [vp, vp, sz, vp]
        L.spec_copy_from_host.restype = i32
        L.spec_lmhead_verify.argtypes = [vp, i32, i64, i64, vp, i32, i32, vp, vp, vp, vp, sz, vp]
        L.spec_lmhead_verify.restype = i32
        L.spec_verify_accept_greedy.argtypes = [vp, i32, i64, i64, vp, i32, i32, vp, vp, vp, i32,
                                                vp, vp, i32, vp, vp, vp, vp, ctypes.c_float, vp,
                                                vp, vp, vp, sz, vp]
        L.spec_verify_accept_greedy.restype = i32
        L.spec_draft_argmax.argtypes = [vp, i32, i64, i64, vp, i32, vp, vp, vp, i32, vp, i32, vp,
                                        i64, vp, vp, vp, sz, vp]
        L.spec_draft_argmax.restype = i32
        L.spec_accept.argtypes = [i32, i32, vp, vp, vp, vp, i64, i32, vp, vp, i64, i64, vp, i32,
                                  vp, vp, vp, vp, vp, sz, vp]
        L.spec_accept.restype = i32
        L.spec_accept_exact.argtypes = [i32, i32, vp, vp, vp, vp, i64, i32, vp, i32, vp, vp, vp,
                                        vp, vp, sz, vp]
        L.spec_accept_exact.restype = i32
        L.spec_accept_filtered.argtypes = [i32, i32, vp, vp, vp, vp, i64, i32, vp, vp, vp, i32,
                                           vp, vp, vp, vp, vp, sz, vp]
        L.spec_accept_filtered.restype = i32
        L.spec_draft_argmax_rows.argtypes = [vp, i32, i64, i64, i64, i64, vp, i32, vp, vp, vp,
                                             i32, vp, i32, vp, i64, vp, vp, vp, sz, vp]
        L.spec_draft_argmax_rows.restype = i32
        L.spec_accept_rows.argtypes = [i32, i32, vp, vp, vp, vp, i64, i32, vp, vp, i64, i64,
                                       i64, i64, vp, i32, vp, vp, vp, vp, vp, sz, vp]
        L.spec_accept_rows.restype = i32
        L.spec_adapt_width.argtypes = [i32, i32, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp]
        L.spec_adapt_width.restype = i32
        L.spec_adapt_width_mirror.argtypes = [i32, i32, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                              vp, vp]
        L.spec_adapt_width_mirror.restype = i32
        L.spec_commit_rollback.argtypes = [i32, ctypes.POINTER(spec_state_desc), vp, vp, i32, vp,
                                           vp]
        L.spec_commit_rollback.restype = i32
        L.spec_lmhead_verify_noalloc.argtypes = [vp, i32, i64, i64, vp, i32, i32, vp, vp, vp, vp]
        L.spec_lmhead_verify_noalloc.restype = i32
        L.spec_noalloc_scratch_bytes.argtypes = []
        L.spec_noalloc_scratch_bytes.restype = sz
        L.spec_noalloc_error_word.argtypes = [vp, vp]
        L.spec_noalloc_error_word.restype = i32
        L.spec_test_verify_stalled.argtypes = [vp, i64, i64, vp, i32, i32, vp, vp, vp,
                                               ctypes.c_uint32, vp, sz, vp]
        L.spec_test_verify_stalled.restype = i32
        pvp = ctypes.POINTER(ctypes.c_void_p)
        L.spec_width_graph_create.argtypes = [i32, vp, i32, pvp, pvp]
        L.spec_width_graph_create.restype = i32
        L.spec_graph_capture_begin.argtypes = [vp, vp]
        L.spec_graph_capture_begin.restype = i32
        L.spec_graph_capture_end.argtypes = [vp]
        L.spec_graph_capture_end.restype = i32
        L.spec_graph_instantiate.argtypes = [vp, pvp]
        L.spec_graph_instantiate.restype = i32
        L.spec_graph_launch.argtypes = [vp, vp]
        L.spec_graph_launch.restype = i32
        L.spec_graph_destroy.argtypes = [vp, vp]
        L.spec_graph_destroy.restype = i32
        _lib = L
    return _lib
