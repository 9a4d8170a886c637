"""The C-ABI library loads without a GPU and exports every entry point that
include/vsd.h declares (no compute calls)."""
import ctypes
import os
import re

from speculative_decoding_block_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "vsd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vsd_[a-z0-9_]+)\s*\(", src)))


def test_header_declarations_are_exported():
    build.build()
    lib = ctypes.CDLL(build.OUT)
    names = _declared()
    assert len(names) >= 19
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    assert sorted(binding.EXPORTS) == _declared()


def test_host_side_errors_without_gpu():
    L = binding.lib()
    assert L.vsd_version().decode().startswith("vsd")
    # NULL arguments are rejected on the host before anything touches a device
    assert L.vsd_quantize_fp8_rowwise(None, 4, 4, None, None, None) == binding.VSD_ERR_ARG
    assert b"NULL" in L.vsd_last_error()
    assert L.vsd_verify_step(None, None, 1, None, None, None, None, None, None) == binding.VSD_ERR_ARG
    assert L.vsd_verify_step_host(None, None, 1, None, None, None, None, None, None) == binding.VSD_ERR_ARG
    cfg = binding.ModelConfig(2, 256, 4, 2, 96, 688, 4096, 1e4, 1e-6, 1, 0, 0, 256)
    h = ctypes.c_void_p()
    assert L.vsd_model_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == binding.VSD_ERR_UNSUPPORTED
    assert b"head_dim" in L.vsd_last_error()
    cfg.head_dim, cfg.n_q = 64, 3
    assert L.vsd_model_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == binding.VSD_ERR_ARG


def test_host_array_checks():
    """The host-buffer step's argument marshalling: int32, contiguous, long
    enough, writeable where the call writes."""
    import numpy as np
    import pytest
    ok = np.zeros(34, dtype=np.int32)
    assert binding._host(ok, "a", 34).value == ok.ctypes.data
    with pytest.raises(TypeError):
        binding._host(ok.astype(np.int64), "a", 34)
    with pytest.raises(TypeError):
        binding._host(np.zeros((4, 9), np.int32)[:, :8], "a", 32)
    with pytest.raises(ValueError):
        binding._host(ok, "a", 35)
    ro = np.zeros(16, dtype=np.int32)
    ro.flags.writeable = False
    assert binding._host(ro, "drafts", 16, writable=False).value == ro.ctypes.data
    with pytest.raises(TypeError):
        binding._host(ro, "seq_lens", 16)


def test_rollback_object_argument_checks_without_gpu():
    """vsd_ssm_create rejects bad shapes on the host, before any device call."""
    L = binding.lib()
    h = ctypes.c_void_p()
    assert L.vsd_ssm_create(4, 2, 128, 64, None) == binding.VSD_ERR_ARG           # NULL out
    assert L.vsd_ssm_create(0, 2, 128, 64, ctypes.byref(h)) == binding.VSD_ERR_ARG  # no requests
    assert L.vsd_ssm_create(4, 2, 128, 16, ctypes.byref(h)) == binding.VSD_ERR_ARG  # window below one block
    assert L.vsd_ssm_create(4, 2, 64, 129, ctypes.byref(h)) == binding.VSD_ERR_ARG  # window above the buffer's cap
    assert L.vsd_ssm_create(4, 2, 96, 64, ctypes.byref(h)) == binding.VSD_ERR_UNSUPPORTED
    assert b"64 or 128" in L.vsd_last_error()
    assert L.vsd_ssm_create(4, 2, 128, 65, ctypes.byref(h)) == binding.VSD_ERR_UNSUPPORTED  # shared memory
    assert b"window 65" in L.vsd_last_error()
    assert not h.value
    assert L.vsd_ssm_verify(None, 1, None, None, None, None, None, None, None) == binding.VSD_ERR_ARG
    assert L.vsd_ssm_commit(None, 1, None, None) == binding.VSD_ERR_ARG
