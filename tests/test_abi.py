"""The C-ABI library loads without a GPU, exports every function that include/sdm.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import subprocess

import pytest

import sparse_memory_linear_key_b300 as sdm


@pytest.fixture(scope="module")
def L():
    from sparse_memory_linear_key_b300 import build
    build.build()
    return sdm.lib()


def test_exports_every_declared_symbol(L):
    names = sdm.exported_names()
    assert len(names) >= 12
    out = subprocess.check_output(["nm", "-D", "--defined-only", sdm.LIB_PATH]).decode()
    defined = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in names:
        assert n in defined, n
        assert hasattr(L, n)
    # nothing else of the library leaks into the dynamic symbol table
    ours = {d for d in defined if d.startswith("sdm_")}
    assert ours == set(names)


def test_version_and_status_strings(L):
    assert sdm.version() == "0.1.0"
    assert "timed" in sdm.status_string(sdm.SDM_ETIMEOUT) or "wait" in sdm.status_string(-4)
    assert sdm.status_string(0) == "SDM_OK"


@pytest.mark.parametrize("cfg,want", [
    ((2048, 480, 256, 64, "bf16"), sdm.SDM_OK),
    ((64, 32, 64, 8, "f32"), sdm.SDM_OK),
    ((3840, 480, 256, 64, "bf16"), sdm.SDM_OK),
    ((2040, 480, 256, 64, "bf16"), sdm.SDM_EUNSUPPORTED),   # d % 16
    ((2048, 480, 256, 48, "bf16"), sdm.SDM_EUNSUPPORTED),   # w not in {8,16,32,64}
    ((2048, 32, 256, 64, "bf16"), sdm.SDM_EUNSUPPORTED),    # w > n_sub
    ((2048, 513, 256, 64, "bf16"), sdm.SDM_EUNSUPPORTED),   # n_sub > 512
    ((2048, 480, 512, 64, "bf16"), sdm.SDM_EUNSUPPORTED),   # dk/2 > 128
    ((2048, 480, 255, 64, "bf16"), sdm.SDM_EUNSUPPORTED),   # odd dk
    ((2048, 480, 256, 64, "f32"), sdm.SDM_EUNSUPPORTED),    # fp32 keys too big for smem
    ((0, 480, 256, 64, "bf16"), sdm.SDM_EINVAL),
])
def test_check_cfg(L, cfg, want):
    assert sdm.check_cfg(sdm.make_cfg(*cfg)) == want


def test_workspace_sizes(L):
    c = sdm.make_cfg(2048, 480, 256, 64, "bf16")
    ntok = 4 * 4096
    ws = sdm.workspace_bytes(c, 4, 4096)
    # q_w, q_r, v (bf16), idx + wsel (int32/fp32), the scan's workspace, half lists
    front = ntok * (2 * 256 * 2 + 2048 * 2 + 128 * 4 * 2) + 2 * ntok * 2 * 64 * 8
    scan = sdm.scan_workspace_bytes(c, 4, 4096)
    assert front + scan <= ws <= front + scan + 8 * 256
    # scan: codes (uint16), four ordering masks (uint64), one progress flag per token
    # and 1 KB row block (4 blocks at d = 2048 bf16), then the forwarding ring (whole
    # 1 KB chunks of up to 64 slots per ring entry, 4 sequences x 4 blocks, 16..256
    # entries)
    small = ntok * (128 * 2 + 32 + 4 * 4)
    smin = sdm.scan_min_workspace_bytes(c, 4, 4096)
    assert small <= smin <= small + 4 * 256
    ring = scan - smin
    assert ring % (16 * 64 * 1024) == 0 and 16 <= ring // (16 * 64 * 1024) <= 256
    assert sdm.address_workspace_bytes(c, ntok) >= 2 * ntok * 2 * 64 * 8
    assert sdm.workspace_bytes(sdm.make_cfg(2048, 480, 256, 63, "bf16"), 1, 1) == 0
    # a single decode step: the ring holds one entry per stream
    assert sdm.scan_workspace_bytes(c, 64, 1) - sdm.scan_min_workspace_bytes(c, 64, 1) == \
        64 * 4 * 64 * 1024


def test_host_validation_before_cuda(L):
    c = sdm.make_cfg(64, 32, 64, 8, "f32")
    P = ctypes.c_void_p
    # null pointers and negative sizes fail with SDM_EINVAL, no device touched
    assert L.sdm_init_bank(ctypes.byref(c), None, None, 2, None) == sdm.SDM_EINVAL
    assert L.sdm_init_bank(ctypes.byref(c), None, None, 0, None) == sdm.SDM_OK
    assert L.sdm_init_bank(ctypes.byref(c), P(16), P(32), -1, None) == sdm.SDM_EINVAL
    assert L.sdm_init_bank(ctypes.byref(c), P(17), P(4096), 1, None) == sdm.SDM_EINVAL  # align
    # overlapping source and destination
    assert L.sdm_init_bank(ctypes.byref(c), P(4096), P(4096), 1, None) == sdm.SDM_EINVAL
    w = sdm.Weights(16, 16, 16, 16, 16)
    assert L.sdm_prefill(ctypes.byref(c), ctypes.byref(w), P(16), P(16), P(16), P(16), P(16),
                         1, 8, None, None, P(256), 16, P(16), None) == sdm.SDM_EWORKSPACE
    assert L.sdm_prefill(ctypes.byref(c), ctypes.byref(w), P(16), P(16), P(16), P(16), P(16),
                         1, 8, None, None, P(255), 1 << 20, P(16), None) == sdm.SDM_EINVAL
    assert L.sdm_scan(ctypes.byref(c), None, None, None, None, None, None, None, 1, 1, None, 0,
                      None, None) == sdm.SDM_EINVAL
    assert L.sdm_scan(ctypes.byref(c), P(16), P(16), P(16), P(16), P(16), P(16), P(16), 1, 4,
                      P(256), 8, P(16), None) == sdm.SDM_EWORKSPACE
    assert L.sdm_address(ctypes.byref(c), P(16), P(16), P(16), P(16), 8, P(16), P(16), P(256), 8,
                         P(16), None) == sdm.SDM_EWORKSPACE
    assert L.sdm_project(ctypes.byref(c), None, P(16), 4, P(16), P(16), P(16), None) == sdm.SDM_EINVAL
    # empty work is a no-op
    assert L.sdm_scan(ctypes.byref(c), None, None, None, None, None, None, None, 0, 5, None, 0,
                      None, None) == sdm.SDM_OK
    # the backward walk: every row is staged by 16-byte copies; offsets within a bank are
    # 32-bit; the workspace holds per-block partial sums and 16-byte slot descriptors
    bw = lambda cc, ptr, ws, nbytes: L.sdm_scan_backward(
        ctypes.byref(cc), *([P(ptr)] * 13), 1, 4, P(ws), nbytes, None)
    need = sdm.scan_backward_workspace_bytes(c, 1, 4)
    assert need == (((64 + 63) // 64) * 4 * (2 * 8 + 2) * 4 + 255) // 256 * 256 + 4 * 8 * 16
    assert bw(c, 24, 256, need) == sdm.SDM_EINVAL                    # misaligned
    assert bw(c, 16, 256, need - 1) == sdm.SDM_EWORKSPACE
    big = sdm.make_cfg(16400, 512, 256, 64, "bf16")                  # N d > 2^32
    assert bw(big, 16, 256, 1 << 40) == sdm.SDM_EUNSUPPORTED


def test_binding_refuses_cpu_tensors(L):
    import torch
    c = sdm.make_cfg(64, 32, 64, 8, "f32")
    M0 = torch.zeros(1024, 64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sdm.sdm_init_bank(c, M0, torch.zeros(1, 1024, 64))
