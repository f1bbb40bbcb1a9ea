"""CPU checks of the C ABI: the library builds and loads, exports every symbol include/spec.h
declares, and rejects bad arguments on the host before touching the GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mtp_speculative_decoding_spec_gb300 import build
    build.build()
    import mtp_speculative_decoding_spec_gb300 as spec
    return spec._abi.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "spec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "spec_lmhead_verify" in names and "spec_commit_rollback" in names
    for n in names:
        assert hasattr(lib, n), n
    import mtp_speculative_decoding_spec_gb300 as spec
    assert set(spec._abi.EXPORTS) == set(names)


def test_status_strings(lib):
    assert lib.spec_status_str(0) == b"SPEC_OK"
    assert lib.spec_status_str(1) == b"SPEC_ERR_INVALID"
    assert lib.spec_status_str(3) == b"SPEC_ERR_CUDA"


def test_struct_layouts_match_the_c_compiler(tmp_path):
    """Sizes and field offsets of the binding's structs equal what a C compiler gives for
    include/spec.h."""
    import shutil
    import subprocess

    import mtp_speculative_decoding_spec_gb300 as spec
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in spec.spec_state_desc._fields_]
    # numpy views of the result structs: (C struct, dtype) with the same field names
    views = [("spec_rowstats", spec.ROWSTATS_DTYPE), ("spec_accept_out", spec.ACCEPT_OUT_DTYPE),
             ("spec_counters", spec.COUNTERS_DTYPE), ("spec_width_state", spec.WIDTH_STATE_DTYPE)]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "spec.h"', "int main(void){",
            'printf("%zu %zu %zu %zu\\n", sizeof(spec_rowstats), sizeof(spec_accept_out), '
            "sizeof(spec_counters), sizeof(spec_state_desc));"]
    for f in fields:
        prog.append(f'printf("%zu\\n", offsetof(spec_state_desc, {f}));')
    for cname, dt in views:
        prog.append(f'printf("%zu\\n", sizeof({cname}));')
        for f in dt.names:
            prog.append(f'printf("%zu\\n", offsetof({cname}, {f}));')
    prog.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    sizes = [int(x) for x in out[:4]]
    assert sizes == [spec.ROWSTATS_BYTES, spec.ACCEPT_OUT_BYTES, spec.COUNTERS_BYTES,
                     ctypes.sizeof(spec.spec_state_desc)]
    offs = [int(x) for x in out[4:4 + len(fields)]]
    assert offs == [getattr(spec.spec_state_desc, f).offset for f in fields]
    rest = [int(x) for x in out[4 + len(fields):]]
    for cname, dt in views:
        assert rest[0] == dt.itemsize, cname
        assert rest[1:1 + len(dt.names)] == [dt.fields[f][1] for f in dt.names], cname
        rest = rest[1 + len(dt.names):]
    assert rest == []


def test_host_validation_without_gpu(lib):
    """Null pointers and out-of-range sizes are rejected before any CUDA call."""
    null = None
    fake = 256  # a 16-byte aligned non-null pointer value; never dereferenced on these paths
    assert lib.spec_lmhead_verify(null, 0, 10, 64, fake, 1, 1, fake, null, fake, fake, 1 << 20,
                                  null) == 1
    assert lib.spec_lmhead_verify(fake, 0, 10, 64, fake, 1, 9, fake, null, fake, fake, 1 << 20,
                                  null) == 1
    assert lib.spec_lmhead_verify(fake, 7, 10, 64, fake, 1, 1, fake, null, fake, fake, 1 << 20,
                                  null) == 1
    assert lib.spec_lmhead_verify(fake + 8, 0, 10, 64, fake, 1, 1, fake, null, fake, fake,
                                  1 << 20, null) == 1
    assert lib.spec_lmhead_verify(fake, 0, 1 << 24, 64, fake, 1, 1, fake, null, fake, fake,
                                  1 << 20, null) == 1
    assert lib.spec_draft_argmax(fake, 0, 10, 64, fake, 9, fake, fake, fake, 0, fake, 1, null,
                                 0, null, null, fake, 1 << 20, null) == 1
    assert lib.spec_accept(0, 3, fake, fake, fake, fake, 10, 4, null, null, 10, 10, fake, 2,
                           fake, fake, fake, null, fake, 1 << 20, null) == 1
    assert lib.spec_accept(1, 8, fake, fake, fake, fake, 10, 4, null, null, 10, 10, fake, 2,
                           fake, fake, fake, null, fake, 1 << 20, null) == 1
    assert lib.spec_accept(1, 3, fake, fake, fake, fake, 10, 4, fake, null, 10, 10, fake, 2,
                           fake, fake, fake, null, fake, 1 << 20, null) == 1
    import mtp_speculative_decoding_spec_gb300 as spec
    d = spec.spec_state_desc()
    d.n_slots = 9
    d.kv_layers = 1
    assert lib.spec_commit_rollback(1, ctypes.byref(d), fake, fake, 0, null, null) == 1
    d.kv_layers = 0
    assert lib.spec_commit_rollback(1, ctypes.byref(d), fake, fake, 5, null, null) == 1
    assert lib.spec_commit_rollback(1, None, fake, fake, 0, null, null) == 1
    # index mode: a recurrent state needs the live-slot array, and nothing else of the state
    d.rec_layers, d.rec_heads, d.rec_dk, d.rec_dv = 2, 2, 4, 4
    assert lib.spec_commit_rollback(1, ctypes.byref(d), fake, fake, spec.SPEC_COMMIT_INDEX,
                                    null, null) == 1
    assert lib.spec_commit_rollback(1, ctypes.byref(d), fake, fake, 3, null, null) == 1


def test_host_validation_of_the_later_entry_points(lib):
    """The exact, filtered, adaptive-width and two-range calls, and the weight formats, reject
    bad arguments before any CUDA call."""
    null, fake = None, 256
    # weight format codes: 0 bf16, 1 fp32, 2 4-bit; anything else is invalid
    assert lib.spec_lmhead_verify(fake, 3, 10, 128, fake, 1, 1, fake, null, fake, fake, 1 << 20,
                                  null) == 1
    assert lib.spec_accept_exact(0, 3, fake, fake, fake, fake, 10, 4, fake, 2, fake, fake, fake,
                                 null, fake, 1 << 20, null) == 1
    # filtered acceptance needs both filter arrays
    assert lib.spec_accept_filtered(1, 3, fake, fake, fake, fake, 10, 4, fake, null, fake, 2,
                                    fake, fake, fake, null, fake, 1 << 20, null) == 1
    assert lib.spec_accept_filtered(1, 3, fake, fake, fake, fake, 10, 4, fake, fake, null, 2,
                                    fake, fake, fake, null, fake, 1 << 20, null) == 1
    # adaptive width: sizes, pointers, and alpha in (0, 1]
    assert lib.spec_adapt_width(0, 7, fake, fake, fake, null, 0.1, fake, fake, null) == 1
    assert lib.spec_adapt_width(1, 8, fake, fake, fake, null, 0.1, fake, fake, null) == 1
    assert lib.spec_adapt_width(1, 7, fake, fake, null, null, 0.1, fake, fake, null) == 1
    assert lib.spec_adapt_width(1, 7, fake, fake, fake, null, 0.0, fake, fake, null) == 1
    assert lib.spec_adapt_width(1, 7, fake, fake, fake, fake, 1.5, fake, fake, null) == 1
    # the fused greedy verify + acceptance: the verify's checks, k_max <= 7, k and out required;
    # a width update (state set) needs cost, k_next and alpha in (0, 1]
    def vag(B, R, k_max, k, out, state=null, cost=null, k_next=null, alpha=0.1):
        return lib.spec_verify_accept_greedy(fake, 0, 10, 128, fake, B, R, fake, null, fake,
                                             k_max, k, fake, -1, out, null, cost, null, alpha,
                                             state, k_next, null, fake, 1 << 20, null)
    assert vag(1, 2, 8, fake, fake) == 1
    assert vag(1, 2, 1, null, fake) == 1
    assert vag(1, 2, 1, fake, null) == 1
    assert vag(2, 8, 1, fake, fake) == 2
    assert vag(1, 2, 1, fake, fake, state=fake) == 1                      # no cost, no k_next
    assert vag(1, 2, 1, fake, fake, state=fake, cost=fake, k_next=fake, alpha=0.0) == 1
    # the mirror entry point: the same checks, and the mirror is required
    assert lib.spec_adapt_width_mirror(1, 7, fake, fake, fake, null, 0.1, fake, fake, null,
                                       null) == 1
    assert lib.spec_adapt_width_mirror(0, 7, fake, fake, fake, null, 0.1, fake, fake, fake,
                                       null) == 1
    assert lib.spec_adapt_width_mirror(1, 7, fake, fake, fake, null, 0.0, fake, fake, fake,
                                       null) == 1
    # width graphs: 1..64 bodies, 1..128 requests, the widths and both outputs required
    import ctypes
    g, bodies = ctypes.c_void_p(), (ctypes.c_void_p * 8)()
    assert lib.spec_width_graph_create(0, fake, 1, ctypes.byref(g), bodies) == 1
    assert lib.spec_width_graph_create(8, fake, 129, ctypes.byref(g), bodies) == 1
    assert lib.spec_width_graph_create(8, null, 1, ctypes.byref(g), bodies) == 1
    assert lib.spec_graph_capture_begin(null, fake) == 1
    assert lib.spec_graph_capture_begin(fake, null) == 1  # the legacy stream cannot capture
    assert lib.spec_graph_instantiate(null, ctypes.byref(g)) == 1
    assert lib.spec_graph_launch(null, null) == 1
    # two-range draft set: the second range may not start inside the first, the set may not be
    # empty; a split set needs tensor-core weights and whole 32-row boxes
    rows = lib.spec_draft_argmax_rows
    # d, h, B, temperature, seed, pos, pos_offset, token_out, token_stride, q_logits, q_stride,
    # q_stats, k_active, workspace, workspace_bytes, stream
    args = (64, fake, 1, fake, fake, fake, 0, fake, 1, null, 0, null, null, fake, 1 << 20, null)
    assert rows(fake, 0, 3072, 3000, 256, *args) == 1
    assert rows(fake, 0, 0, 0, 0, *args) == 1
    assert rows(fake, 1, 3072, 3840, 256, *args) == 2
    assert rows(fake, 0, 3000, 3840, 256, *args) == 2
    assert lib.spec_accept_rows(1, 3, fake, fake, fake, fake, 4096, 4, fake, fake, 3072, 3000,
                                256, 3328, fake, 2, fake, fake, fake, null, fake, 1 << 20,
                                null) == 1
    # the allocation-free entry point's error-word copy needs a destination
    assert lib.spec_noalloc_error_word(null, null) == 1
    # the stalled-producer test call: a wait limit in [1 us, 1 s], at most 8 rows in total
    st = lib.spec_test_verify_stalled
    assert st(fake, 4096, 256, fake, 1, 4, fake, null, fake, 0, fake, 1 << 20, null) == 1
    assert st(fake, 4096, 256, fake, 1, 4, fake, null, fake, 1000001, fake, 1 << 20, null) == 1
    assert st(fake, 4096, 256, fake, 3, 4, fake, null, fake, 1000, fake, 1 << 20, null) == 1
    assert st(fake, 4096, 256, fake, 1, 4, fake, null, null, 1000, fake, 1 << 20, null) == 1


def test_empty_inputs_are_rejected(lib):
    """Zero requests, zero rows, an empty vocabulary or hidden size: SPEC_ERR_INVALID from every
    entry point, before any CUDA call (nothing is enqueued for an empty batch)."""
    null, fake = None, 256
    verify = lib.spec_lmhead_verify
    for V, d, B, R in ((0, 64, 1, 1), (10, 0, 1, 1), (10, 64, 0, 1), (10, 64, 1, 0),
                       (-5, 64, 1, 1), (10, 64, -1, 1)):
        assert verify(fake, 0, V, d, fake, B, R, fake, null, fake, fake, 1 << 20, null) == 1
        assert lib.spec_lmhead_verify_noalloc(fake, 0, V, d, fake, B, R, fake, null, fake,
                                              null) == 1
    for V, d, B in ((0, 64, 1), (10, 0, 1), (10, 64, 0)):
        assert lib.spec_draft_argmax(fake, 0, V, d, fake, B, fake, fake, fake, 0, fake, 1, null,
                                     0, null, null, fake, 1 << 20, null) == 1
    for B, V, R in ((0, 10, 4), (1, 0, 4), (1, 10, 0)):
        assert lib.spec_accept(B, 3, fake, fake, fake, fake, V, R, null, null, 10, 10, fake, 2,
                               fake, fake, fake, null, fake, 1 << 20, null) == 1
        assert lib.spec_accept_exact(B, 3, fake, fake, fake, fake, V, R, fake, 2, fake, fake,
                                     fake, null, fake, 1 << 20, null) == 1
        assert lib.spec_accept_filtered(B, 3, fake, fake, fake, fake, V, R, fake, fake, fake, 2,
                                        fake, fake, fake, null, fake, 1 << 20, null) == 1
    import mtp_speculative_decoding_spec_gb300 as spec
    d = spec.spec_state_desc()
    d.n_slots = 9
    assert lib.spec_commit_rollback(0, ctypes.byref(d), fake, fake, 0, null, null) == 1
    assert lib.spec_workspace_bytes(0, 1) == 0 and lib.spec_workspace_bytes(10, 0) == 0


def test_binding_raises_on_error(lib):
    import mtp_speculative_decoding_spec_gb300 as spec
    with pytest.raises(spec.SpecError) as e:
        spec._check("spec_accept", 1)
    assert e.value.status == 1 and "SPEC_ERR_INVALID" in str(e.value)


def test_no_cpu_fallback_in_product_package():
    """The product package never imports the oracle or computes on the host."""
    pkg = os.path.join(ROOT, "mtp_speculative_decoding_spec_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "oracle" not in src, f
            assert "import numpy" not in src or f == "_abi.py", f


# threads per block of each kernel, as launched by abi.cu / gemv.cu
_BLOCK_THREADS = {"gemv_rows_kernel": 16 * 32, "gemv_tc_kernel": 8 * 32, "gemv_q4_kernel": 16 * 32, "gemm_rows_tc_kernel": 10 * 32,
                  "gemm_rows_combine_kernel": 256, "accept_kernel": 256,
                  "commit_index_kernel": 256, "commit_snapshot_kernel": 256,
                  "commit_replay_kernel": 128, "adapt_width_kernel": 128,
                  "width_select_kernel": 32, "copy_from_host_kernel": 256}


def test_register_budget_per_sub_partition(lib):
    """Each SM has four sub-partitions with 16K registers each and a block's warps are spread
    round-robin over them, so regs/thread (allocated in multiples of 8) times 32 times the warps
    on the fullest sub-partition must fit in 16,384 -- or the launch fails. Also: no spills."""
    import glob
    logs = glob.glob(os.path.join(ROOT, "mtp_speculative_decoding_spec_gb300", "_build",
                                  "*.ptxas.log"))
    assert logs, "build did not record ptxas output"
    seen = 0
    for path in logs:
        name = None
        for line in open(path):
            m = re.search(r"Compiling entry function '(\w+)'", line)
            if m:
                name = m.group(1)
            m = re.search(r"(\d+) bytes spill stores", line)
            if m and name:
                assert int(m.group(1)) == 0, f"{name} spills"
            m = re.search(r"Used (\d+) registers", line)
            if m and name:
                regs = int(m.group(1))
                base = next(k for k in _BLOCK_THREADS if k in name)
                warps = _BLOCK_THREADS[base] // 32
                per_sp = -(-warps // 4)
                alloc = -(-regs // 8) * 8
                assert alloc * 32 * per_sp <= 16384, (name, regs, warps)
                seen += 1
    assert seen >= 10


def _header_prototypes():
    """(name, return type, [parameter types]) of every function include/spec.h declares."""
    src = open(os.path.join(ROOT, "include", "spec.h")).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    protos = []
    for m in re.finditer(r"([A-Za-z_][\w \*]*?)\b(spec_\w+)\s*\(([^;{]*?)\)\s*;", src):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        if ret.startswith("typedef"):
            continue
        plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        types = [re.sub(r"\s*\b\w+$", "", p) if not p.endswith("*") else p for p in plist]
        protos.append((name, ret, types))
    return protos


def _ctype_of(ctype):
    """The ctypes argument kind a C parameter type needs: (size in bytes, pointer, float)."""
    t = " ".join(ctype.replace("*", " * ").split())
    if "*" in t:
        return (ctypes.sizeof(ctypes.c_void_p), True, False)
    base = t.replace("const ", "")
    sizes = {"int32_t": 4, "uint32_t": 4, "int64_t": 8, "size_t": ctypes.sizeof(ctypes.c_size_t),
             "float": 4, "spec_dtype": 4, "spec_status": 4}
    if base == "spec_stream_t":
        return (ctypes.sizeof(ctypes.c_void_p), True, False)
    return (sizes[base], False, base == "float")


def _kind(ct):
    is_ptr = ct in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(ct, "_type_") and \
        isinstance(ct._type_, type)
    return (ctypes.sizeof(ct), bool(is_ptr), ct is ctypes.c_float)


def test_binding_signatures_match_the_header(lib):
    """Every declared function's ctypes argtypes and restype agree with include/spec.h in count,
    size, pointer-ness and floating point, so the binding passes each argument as C expects."""
    protos = _header_prototypes()
    names = {n for n, _, _ in protos}
    import mtp_speculative_decoding_spec_gb300._abi as abi
    assert names == set(abi.EXPORTS)
    for name, ret, params in protos:
        fn = getattr(lib, name)
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), params)
        for i, (ct, p) in enumerate(zip(fn.argtypes, params)):
            assert _kind(ct) == _ctype_of(p), (name, i, p, ct)
        if ret.endswith("*"):
            assert fn.restype in (ctypes.c_char_p, ctypes.c_void_p), name
        else:
            assert ctypes.sizeof(fn.restype) == _ctype_of(ret)[0], (name, ret, fn.restype)
