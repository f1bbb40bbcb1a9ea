"""Host transfers inside the chain of kernels (spec_copy_from_host, spec_host_alias): copies
from pinned host memory are bitwise exact at several sizes, invalid sources and sizes are
refused before anything is enqueued, and an acceptance that writes its result through a host
alias writes the same bytes it writes to device memory."""

import numpy as np
import pytest

from synth import configs, gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import dev, ensure_built, to_dev, to_np, workspace, zeros_bytes  # noqa: E402
import mtp_speculative_decoding_spec_gb300 as spec  # noqa: E402


@pytest.mark.parametrize("nbytes", [16, 10_256, 1 << 20, (1 << 20) + 48])
def test_copy_from_host_is_exact(nbytes):
    ensure_built()
    rng = np.random.default_rng(nbytes)
    src = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dst = torch.zeros(nbytes + 64, dtype=torch.uint8, device=dev())
    spec.spec_copy_from_host(dst, src, nbytes)
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    assert got[:nbytes].tobytes() == src.numpy().tobytes()
    assert not got[nbytes:].any()  # nothing written past the end


def test_copy_from_host_refuses_bad_arguments():
    ensure_built()
    lib = spec._abi.lib()
    stream = torch.cuda.current_stream().cuda_stream
    pinned = torch.zeros(256, dtype=torch.uint8).pin_memory()
    pageable = np.zeros(256, dtype=np.uint8)
    d = torch.zeros(256, dtype=torch.uint8, device=dev())
    assert lib.spec_copy_from_host(d.data_ptr(), pageable.ctypes.data, 64, stream) == 1
    assert lib.spec_copy_from_host(d.data_ptr(), pinned.data_ptr(), 40, stream) == 1  # not x16
    assert lib.spec_copy_from_host(d.data_ptr() + 4, pinned.data_ptr(), 64, stream) == 1
    assert lib.spec_copy_from_host(d.data_ptr(), pinned.data_ptr() + 8, 64, stream) == 1
    assert lib.spec_copy_from_host(d.data_ptr(), d.data_ptr(), 64, stream) == 1  # not host
    assert lib.spec_copy_from_host(d.data_ptr(), pinned.data_ptr(), 0, stream) == 0
    with pytest.raises(spec.SpecError):
        spec.spec_host_alias(pageable.ctypes.data)
    with pytest.raises(spec.SpecError):
        spec.spec_host_alias(d)
    assert spec.spec_host_alias(pinned) != 0
    torch.cuda.synchronize()


def test_accept_result_through_a_host_alias():
    """Verify + acceptance at the sampled k = 3 shape of C0, once with the result in device
    memory and once through the host alias of pinned memory: the same bytes."""
    ensure_built()
    cfg = configs.get(0)
    W = gen.lm_weights(cfg)
    Wd = to_dev(W)
    B, k = 2, cfg.k
    R = k + 1
    rng = np.random.default_rng(77)
    H = gen.encode(rng.standard_normal((B * R, cfg.d), dtype=np.float32), cfg.wdtype)
    ws = workspace(cfg.V, B)
    logits = torch.zeros((B * R, cfg.V), dtype=torch.float32, device=dev())
    stats = zeros_bytes(B * R * spec.ROWSTATS_BYTES)
    temps = torch.tensor([1.0, 0.0], dtype=torch.float32, device=dev())
    spec.spec_lmhead_verify(Wd, spec.SPEC_F32 if cfg.wdtype == "f32" else spec.SPEC_BF16, cfg.V,
                            cfg.d, to_dev(H), B, R, temps, logits, stats, ws)
    drafts = to_dev(rng.integers(0, cfg.V, (B, k), dtype=np.int32))
    kk = to_dev(np.full(B, k, dtype=np.int32))
    seeds = to_dev(np.array([5, 6], dtype=np.uint64))
    pos = to_dev(np.array([100, 200], dtype=np.int64))
    out_dev = zeros_bytes(B * spec.ACCEPT_OUT_BYTES)
    out_host = torch.zeros(B * spec.ACCEPT_OUT_BYTES, dtype=torch.uint8).pin_memory()

    def accept(out):
        spec.spec_accept(B, k, kk, drafts, logits, stats, cfg.V, R, None, None, cfg.Vd, cfg.Vd,
                         temps, cfg.eos_id, seeds, pos, out, None, ws)

    accept(out_dev)
    accept(spec.spec_host_alias(out_host))
    torch.cuda.synchronize()
    assert out_host.numpy().tobytes() == to_np(out_dev).tobytes()
    o = out_host.numpy().view(spec.ACCEPT_OUT_DTYPE)
    assert (o["status"] == 0).all() and (o["n_emit"] >= 1).all()
