"""Device-side error paths and launch order, on the GPU, with test-only
kernels of tests/gpu_probes/probe_kernels.cu (built here into a library of
their own; nothing of it is in libgdn.so).

- A bounded mbarrier wait that runs out: a probe kernel waits with the
  library's wait helper and a poll limit of 16 polls on a barrier that
  nothing signals, reporting into libgdn's error word (gdn_device_error_word).
  gdn_check_device_error must return GDN_ERR_TIMEOUT with the wait site in
  its message, and clear the word; the first report wins.
- Programmatic launch order: gdn_forward's kernel may be scheduled while the
  previous kernel runs, so a previous kernel that triggers its dependents at
  once and writes the state_in pointer array only later must still be seen
  whole. The result must equal the same call after a device synchronisation
  bit for bit.
"""
import ctypes
import os
import subprocess

import pytest
import torch

from gated_delta_net_02_gb300 import inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


@pytest.fixture(scope="module")
def probe(gdn, tmp_path_factory):
    from gated_delta_net_02_gb300 import build
    out = str(tmp_path_factory.mktemp("probe") / "libgdn_probe.so")
    cmd = [build._nvcc()] + build.NVCC_FLAGS + [
        "-shared", os.path.join(ROOT, "tests", "gpu_probes", "probe_kernels.cu"), "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lib = ctypes.CDLL(out)
    lib.gdn_probe_timeout.restype = ctypes.c_int
    lib.gdn_probe_timeout.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint,
                                      ctypes.c_void_p]
    lib.gdn_probe_delayed_copy.restype = ctypes.c_int
    lib.gdn_probe_delayed_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                           ctypes.c_ulonglong, ctypes.c_void_p]
    return lib


def test_bounded_wait_timeout_is_reported_and_cleared(gdn, probe):
    gdn.gdn_check_device_error()                 # start from a clear word
    word = gdn.gdn_device_error_word()
    assert word != 0
    assert probe.gdn_probe_timeout(word, 54, 16, None) == 0
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_check_device_error()
    assert e.value.status == gdn.GDN_ERR_TIMEOUT
    assert "site 54: chunk scan, D tile" in str(e.value)
    gdn.gdn_check_device_error()                 # cleared: no error now


def test_first_timeout_report_wins(gdn, probe):
    gdn.gdn_check_device_error()
    word = gdn.gdn_device_error_word()
    assert probe.gdn_probe_timeout(word, 77, 16, None) == 0
    assert probe.gdn_probe_timeout(word, 11, 16, None) == 0
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_check_device_error()
    assert e.value.status == gdn.GDN_ERR_TIMEOUT
    assert "site 77" in str(e.value) and "site 11" not in str(e.value)
    gdn.gdn_check_device_error()


def test_library_calls_work_after_a_timeout(gdn, probe):
    # the context stays usable: a decode call right after a reported timeout
    gdn.gdn_check_device_error()
    assert probe.gdn_probe_timeout(gdn.gdn_device_error_word(), 23, 16, None) == 0
    with pytest.raises(gdn.GDNError):
        gdn.gdn_check_device_error()
    b = inputs.make_batch(400, [1] * 4, 2, 128, 128, n_slots=1)
    from _helpers import gpu_forward, oracle_run, rel_l2
    out, _ = gpu_forward(b)
    o_ref, _, _ = oracle_run(b)
    assert rel_l2(out.double().cpu().numpy(), o_ref) <= 5e-3


def test_pointer_array_written_by_an_early_triggering_kernel(gdn, probe):
    """A verify call (T = 8, K = 8) whose state_in array is written by the
    kernel right before it, which triggers its dependents at its start and
    writes only after a 50 us delay. The array first holds pointers to a
    decoy state bank; the call must use the bank the previous kernel wrote."""
    N, T, H, D, K = 16, 8, 4, 128, 8
    b = inputs.make_batch(401, [T] * N, H, D, D, n_slots=K)
    dev = {n: getattr(b, n).cuda().contiguous() for n in ("q", "k", "v", "g", "beta", "state")}
    decoy = torch.randn_like(dev["state"])
    good = gdn.state_ptr_array(gdn.per_seq_state_ptrs(dev["state"], N), "cuda")
    bad = gdn.state_ptr_array(gdn.per_seq_state_ptrs(decoy, N), "cuda")
    shape = gdn.gdn_shape(N, T, H, D, D, gdn.GDN_BF16, b.scale)
    stream = torch.cuda.Stream()

    def call(ptrs, out, slots):
        gdn.gdn_forward(shape, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], ptrs, slots,
                        out, K, "gda", stream)

    ref_out = torch.empty(N * T, H, D, device="cuda")
    ref_slots = torch.empty(N, K, H, D, D, device="cuda")
    torch.cuda.synchronize()
    call(good, ref_out, ref_slots)
    torch.cuda.synchronize()
    for rep in range(3):
        ptrs = bad.clone()
        out = torch.full_like(ref_out, float("nan"))
        slots = torch.full_like(ref_slots, float("nan"))
        torch.cuda.synchronize()
        assert probe.gdn_probe_delayed_copy(good.data_ptr(), ptrs.data_ptr(), N, 50_000,
                                            stream.cuda_stream) == 0
        call(ptrs, out, slots)
        stream.synchronize()
        gdn.gdn_check_device_error(stream)
        assert torch.equal(out, ref_out), f"repeat {rep}"
        assert torch.equal(slots, ref_slots), f"repeat {rep}"
