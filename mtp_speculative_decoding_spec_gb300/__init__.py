"""Python binding of libspec.so: the per-cycle verify step of MTP speculative decoding on a
GB300 (sm_103a).

Each function has the name and argument order of the C call in include/spec.h and only
marshals arguments: torch tensors (device memory) become raw pointers, the stream defaults to
torch's current stream, and a non-zero spec_status raises SpecError. Every step of the path
runs in the library's CUDA kernels; nothing here computes, and nothing falls back to the CPU.
"""

from . import _abi
from ._abi import (ACCEPT_OUT_DTYPE, COUNTERS_DTYPE, REQ_BAD_FILTER, REQ_BAD_K,  # noqa: F401
                   REQ_BAD_TOKEN,
                   REQ_KV_OVERFLOW, REQ_NO_LOGITS, REQ_NONFINITE, REQ_OK, ROWSTATS_DTYPE,
                   SPEC_BF16, SPEC_COMMIT_INDEX, SPEC_COMMIT_REPLAY, SPEC_COMMIT_SNAPSHOT, SPEC_F32,
                   SPEC_Q4A32,
                   WIDTH_STATE_DTYPE, spec_state_desc)

ROWSTATS_BYTES = ROWSTATS_DTYPE.itemsize
ACCEPT_OUT_BYTES = ACCEPT_OUT_DTYPE.itemsize
COUNTERS_BYTES = COUNTERS_DTYPE.itemsize
WIDTH_STATE_BYTES = WIDTH_STATE_DTYPE.itemsize


class SpecError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        msg = _abi.lib().spec_status_str(status).decode()
        super().__init__(f"{name} returned {msg} ({status})")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, st):
    if st != 0:
        raise SpecError(name, st)


def spec_workspace_bytes(V, max_batch):
    return int(_abi.lib().spec_workspace_bytes(int(V), int(max_batch)))


def spec_batched_supported():
    return bool(_abi.lib().spec_batched_supported())


def spec_host_alias(host):
    """Device address (int) of pinned, mapped host memory (a pinned tensor or an address)."""
    import ctypes
    out = ctypes.c_void_p()
    _check("spec_host_alias", _abi.lib().spec_host_alias(_ptr(host), ctypes.byref(out)))
    return int(out.value)


def spec_copy_from_host(dst, src_host, nbytes, stream=None):
    _check("spec_copy_from_host", _abi.lib().spec_copy_from_host(
        _ptr(dst), _ptr(src_host), int(nbytes), _stream(stream)))


def spec_lmhead_verify(W, wdt, V, d, H, B, R, temperature, logits, stats, workspace,
                       stream=None):
    _check("spec_lmhead_verify", _abi.lib().spec_lmhead_verify(
        _ptr(W), wdt, V, d, _ptr(H), B, R, _ptr(temperature), _ptr(logits), _ptr(stats),
        _ptr(workspace), _nbytes(workspace), _stream(stream)))


def spec_verify_accept_greedy(W, wdt, V, d, H, B, R, temperature, logits, stats, k_max, k,
                              drafts, eos_id, out, counters, workspace, stream=None, cost=None,
                              cycle_cost=None, alpha=0.1, state=None, k_next=None,
                              k_mirror=None):
    """Verify + greedy acceptance in one launch; with `state` also the width update of
    spec_adapt_width_mirror (k_mirror: a device-writable address or a tensor)."""
    _check("spec_verify_accept_greedy", _abi.lib().spec_verify_accept_greedy(
        _ptr(W), wdt, V, d, _ptr(H), B, R, _ptr(temperature), _ptr(logits), _ptr(stats), k_max,
        _ptr(k), _ptr(drafts), eos_id, _ptr(out), _ptr(counters), _ptr(cost), _ptr(cycle_cost),
        float(alpha), _ptr(state), _ptr(k_next), _ptr(k_mirror), _ptr(workspace),
        _nbytes(workspace), _stream(stream)))


def spec_draft_argmax(W, wdt, V_draft, d, h, B, temperature, seed, pos, pos_offset, token_out,
                      token_stride, q_logits, q_stride, q_stats, k_active, workspace,
                      stream=None):
    _check("spec_draft_argmax", _abi.lib().spec_draft_argmax(
        _ptr(W), wdt, V_draft, d, _ptr(h), B, _ptr(temperature), _ptr(seed), _ptr(pos),
        pos_offset, _ptr(token_out), token_stride, _ptr(q_logits), q_stride, _ptr(q_stats),
        _ptr(k_active), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def spec_draft_argmax_rows(W, wdt, n_low, hi_first, n_high, d, h, B, temperature, seed, pos,
                           pos_offset, token_out, token_stride, q_logits, q_stride, q_stats,
                           k_active, workspace, stream=None):
    _check("spec_draft_argmax_rows", _abi.lib().spec_draft_argmax_rows(
        _ptr(W), wdt, n_low, hi_first, n_high, d, _ptr(h), B, _ptr(temperature), _ptr(seed),
        _ptr(pos), pos_offset, _ptr(token_out), token_stride, _ptr(q_logits), q_stride,
        _ptr(q_stats), _ptr(k_active), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def spec_accept_rows(B, k_max, k, drafts, logits, stats, V, R, q_logits, q_stats, n_low,
                     hi_first, n_high, q_stride, temperature, eos_id, seed, pos_base, out,
                     counters, workspace, stream=None):
    _check("spec_accept_rows", _abi.lib().spec_accept_rows(
        B, k_max, _ptr(k), _ptr(drafts), _ptr(logits), _ptr(stats), V, R, _ptr(q_logits),
        _ptr(q_stats), n_low, hi_first, n_high, q_stride, _ptr(temperature), eos_id, _ptr(seed),
        _ptr(pos_base), _ptr(out), _ptr(counters), _ptr(workspace), _nbytes(workspace),
        _stream(stream)))


def spec_accept(B, k_max, k, drafts, logits, stats, V, R, q_logits, q_stats, V_draft, q_stride,
                temperature, eos_id, seed, pos_base, out, counters, workspace, stream=None):
    _check("spec_accept", _abi.lib().spec_accept(
        B, k_max, _ptr(k), _ptr(drafts), _ptr(logits), _ptr(stats), V, R, _ptr(q_logits),
        _ptr(q_stats), V_draft, q_stride, _ptr(temperature), eos_id, _ptr(seed), _ptr(pos_base),
        _ptr(out), _ptr(counters), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def spec_adapt_width(B, k_max, out, k_used, cost, cycle_cost, alpha, state, k_next,
                     stream=None):
    _check("spec_adapt_width", _abi.lib().spec_adapt_width(
        B, k_max, _ptr(out), _ptr(k_used), _ptr(cost), _ptr(cycle_cost), float(alpha),
        _ptr(state), _ptr(k_next), _stream(stream)))


def spec_adapt_width_mirror(B, k_max, out, k_used, cost, cycle_cost, alpha, state, k_next,
                            k_mirror, stream=None):
    """k_mirror: a device-writable address (an int from spec_host_alias) or a tensor."""
    _check("spec_adapt_width_mirror", _abi.lib().spec_adapt_width_mirror(
        B, k_max, _ptr(out), _ptr(k_used), _ptr(cost), _ptr(cycle_cost), float(alpha),
        _ptr(state), _ptr(k_next), _ptr(k_mirror), _stream(stream)))


def spec_width_graph_create(n_bodies, k_next, B):
    """Returns (graph, [body graphs]) as integers (see include/spec.h)."""
    import ctypes
    g = ctypes.c_void_p()
    bodies = (ctypes.c_void_p * n_bodies)()
    _check("spec_width_graph_create", _abi.lib().spec_width_graph_create(
        n_bodies, _ptr(k_next), B, ctypes.byref(g), bodies))
    return g.value, [bodies[i] for i in range(n_bodies)]


def spec_graph_capture_begin(body, stream):
    _check("spec_graph_capture_begin", _abi.lib().spec_graph_capture_begin(body,
                                                                           _stream(stream)))


def spec_graph_capture_end(stream):
    _check("spec_graph_capture_end", _abi.lib().spec_graph_capture_end(_stream(stream)))


def spec_graph_instantiate(graph):
    import ctypes
    e = ctypes.c_void_p()
    _check("spec_graph_instantiate", _abi.lib().spec_graph_instantiate(graph, ctypes.byref(e)))
    return e.value


def spec_graph_launch(exec_, stream=None):
    _check("spec_graph_launch", _abi.lib().spec_graph_launch(exec_, _stream(stream)))


def spec_graph_destroy(graph, exec_):
    _check("spec_graph_destroy", _abi.lib().spec_graph_destroy(graph, exec_))


def spec_accept_exact(B, k_max, k, drafts, logits, stats, V, R, temperature, eos_id, seed,
                      pos_base, out, counters, workspace, stream=None):
    _check("spec_accept_exact", _abi.lib().spec_accept_exact(
        B, k_max, _ptr(k), _ptr(drafts), _ptr(logits), _ptr(stats), V, R, _ptr(temperature),
        eos_id, _ptr(seed), _ptr(pos_base), _ptr(out), _ptr(counters), _ptr(workspace),
        _nbytes(workspace), _stream(stream)))


def spec_accept_filtered(B, k_max, k, drafts, logits, stats, V, R, temperature, top_k, top_p,
                         eos_id, seed, pos_base, out, counters, workspace, stream=None):
    _check("spec_accept_filtered", _abi.lib().spec_accept_filtered(
        B, k_max, _ptr(k), _ptr(drafts), _ptr(logits), _ptr(stats), V, R, _ptr(temperature),
        _ptr(top_k), _ptr(top_p), eos_id, _ptr(seed), _ptr(pos_base), _ptr(out), _ptr(counters),
        _ptr(workspace), _nbytes(workspace), _stream(stream)))


def spec_commit_rollback(B, st, acc, k, mode, commit_status=None, stream=None):
    """``st`` is a ``spec_state_desc`` (host struct of device pointers)."""
    import ctypes
    _check("spec_commit_rollback", _abi.lib().spec_commit_rollback(
        B, ctypes.byref(st), _ptr(acc), _ptr(k), mode, _ptr(commit_status), _stream(stream)))


def spec_lmhead_verify_noalloc(W, wdt, V, d, H, B, R, temperature, logits, stats, stream=None):
    """spec_lmhead_verify without a workspace: for callers that cannot allocate device memory
    (the library's fixed scratch array is used instead; see include/spec.h)."""
    _check("spec_lmhead_verify_noalloc", _abi.lib().spec_lmhead_verify_noalloc(
        _ptr(W), wdt, V, d, _ptr(H), B, R, _ptr(temperature), _ptr(logits), _ptr(stats),
        _stream(stream)))


def spec_noalloc_scratch_bytes():
    return int(_abi.lib().spec_noalloc_scratch_bytes())


def spec_noalloc_error_word(error_out, stream=None):
    """Enqueue a copy of spec_lmhead_verify_noalloc's error word into ``error_out`` (a 4-byte
    device or pinned host tensor)."""
    _check("spec_noalloc_error_word", _abi.lib().spec_noalloc_error_word(
        _ptr(error_out), _stream(stream)))


def spec_test_verify_stalled(W, V, d, H, B, R, temperature, logits, stats, wait_limit_us,
                             workspace, stream=None):
    """Failure-detection test of the bounded waits: the fp32 verify with a producer that
    issues nothing (see include/spec.h)."""
    _check("spec_test_verify_stalled", _abi.lib().spec_test_verify_stalled(
        _ptr(W), V, d, _ptr(H), B, R, _ptr(temperature), _ptr(logits), _ptr(stats),
        int(wait_limit_us), _ptr(workspace), _nbytes(workspace), _stream(stream)))
