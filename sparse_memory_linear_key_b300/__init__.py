"""Python binding of libsdm.so, the B300 (sm_103a) Sparse Delta Memory layer library.

Argument marshalling only: every function below checks that it got device tensors of
the right dtype and shape, takes their pointers and calls the C entry point of the
same name (include/sdm.h). All arithmetic runs in the CUDA kernels of libsdm.so; there
is no CPU path. If libsdm.so is missing, importing the functions raises.

Layouts (row-major, contiguous): x [B, T, d]; alpha, beta [B, T] fp32; banks
[B, N, d]; y [B, T, d] fp32; idx [B*T, 2, w] int32; wsel [B*T, 2, w] fp32.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libsdm.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "sdm.h")

SDM_OK, SDM_EINVAL, SDM_EUNSUPPORTED, SDM_ECUDA = 0, -1, -2, -3
SDM_ETIMEOUT, SDM_EWORKSPACE, SDM_ERANGE = -4, -5, -6
SDM_F32, SDM_BF16 = 0, 1


class SdmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s: %s" % (what, status_string(code) if _lib is not None else code))


class Cfg(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("n_sub", ctypes.c_int), ("dk", ctypes.c_int),
                ("w", ctypes.c_int), ("dtype", ctypes.c_int)]

    @property
    def N(self) -> int:
        return self.n_sub * self.n_sub

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == SDM_BF16 else torch.float32


class Weights(ctypes.Structure):
    _fields_ = [("W_qw", ctypes.c_void_p), ("W_qr", ctypes.c_void_p), ("W_v", ctypes.c_void_p),
                ("K1", ctypes.c_void_p), ("K2", ctypes.c_void_p)]


_lib = None


def exported_names():
    """Function names declared in include/sdm.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^SDM_API\s+(?:const\s+)?[a-z_0-9]+\*?\s+\**(sdm_[a-z_0-9]+)\s*\(",
                                 text, re.M)))


def lib():
    """Load libsdm.so (built in-tree). Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libsdm.so not found at %s; build it with "
                              "`python -m sparse_memory_linear_key_b300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, I, L64, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        CP = ctypes.POINTER(Cfg)
        WP = ctypes.POINTER(Weights)
        sig = {
            "sdm_status_string": ([I], ctypes.c_char_p),
            "sdm_version": ([], ctypes.c_char_p),
            "sdm_check_cfg": ([CP], I),
            "sdm_workspace_bytes": ([CP, I, I], S),
            "sdm_address_workspace_bytes": ([CP, L64], S),
            "sdm_scan_workspace_bytes": ([CP, I, I], S),
            "sdm_scan_min_workspace_bytes": ([CP, I, I], S),
            "sdm_init_bank": ([CP, P, P, I, P], I),
            "sdm_project": ([CP, WP, P, L64, P, P, P, P], I),
            "sdm_address": ([CP, P, P, P, P, L64, P, P, P, S, P, P], I),
            "sdm_scan": ([CP, P, P, P, P, P, P, P, I, I, P, S, P, P], I),
            "sdm_scan_prepare": ([CP, P, I, I, P, S, P, P], I),
            "sdm_scan_run": ([CP, P, P, P, P, P, P, P, I, I, P, S, P, P], I),
            "sdm_scan_noalloc": ([CP, P, P, P, P, P, P, P, I, I, P, P], I),
            "sdm_scan_run_diag": ([CP, P, P, P, P, P, P, P, I, I, P, S, ctypes.c_longlong,
                                   ctypes.c_longlong, P, P], I),
            "sdm_prefill": ([CP, WP, P, P, P, P, P, I, I, P, P, P, S, P, P], I),
            "sdm_decode_step": ([CP, WP, P, P, P, P, P, I, P, P, P, S, P, P], I),
            "sdm_first_touch_bytes": ([CP, I], S),
            "sdm_first_touch": ([CP, P, I, I, P, P], I),
            "sdm_scan_run_m0": ([CP, P, P, P, P, P, P, P, P, P, I, I, P, S, P, P], I),
            "sdm_fill_untouched": ([CP, P, P, P, I, I, P], I),
            "sdm_prefill_m0_workspace_bytes": ([CP, I, I], S),
            "sdm_prefill_m0": ([CP, WP, P, P, P, P, P, P, I, I, P, P, P, S, P, P], I),
            "sdm_gdn_dense_scan": ([CP, P, P, P, L64, P, P, P, P, P, I, I, P], I),
            "sdm_tape_bytes": ([CP, I, I], S),
            "sdm_address_backward_workspace_bytes": ([CP, L64], S),
            "sdm_project_backward_workspace_bytes": ([CP, L64], S),
            "sdm_project_backward": ([CP, WP, P, L64, P, P, P, P, P, P, P, P, S, P], I),
            "sdm_address_backward": ([CP, P, P, P, P, L64, P, P, P, P, P, P, P, P, S, P], I),
            "sdm_scan_run_train": ([CP, P, P, P, P, P, P, P, P, P, I, I, P, S, P, P, P], I),
            "sdm_scan_backward_workspace_bytes": ([CP, I, I], S),
            "sdm_scan_backward": ([CP, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, P, S, P], I),
            "sdm_slot_counts": ([CP, P, I, I, I, I, I, P, P], I),
            "sdm_slot_overlap_workspace_bytes": ([CP, I], S),
            "sdm_slot_overlap": ([CP, P, I, I, I, I, I, I, P, P, S, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().sdm_status_string(int(code)).decode()


def version() -> str:
    return lib().sdm_version().decode()


def make_cfg(d: int, n_sub: int, dk: int, w: int, dtype) -> Cfg:
    if isinstance(dtype, torch.dtype):
        dtype = SDM_BF16 if dtype == torch.bfloat16 else SDM_F32
    elif isinstance(dtype, str):
        dtype = SDM_BF16 if dtype == "bf16" else SDM_F32
    return Cfg(d, n_sub, dk, w, int(dtype))


def check_cfg(cfg: Cfg) -> int:
    return lib().sdm_check_cfg(ctypes.byref(cfg))


def workspace_bytes(cfg: Cfg, B: int, T: int) -> int:
    return int(lib().sdm_workspace_bytes(ctypes.byref(cfg), B, T))


def address_workspace_bytes(cfg: Cfg, ntok: int) -> int:
    return int(lib().sdm_address_workspace_bytes(ctypes.byref(cfg), ntok))


def scan_workspace_bytes(cfg: Cfg, B: int, T: int) -> int:
    return int(lib().sdm_scan_workspace_bytes(ctypes.byref(cfg), B, T))


def scan_min_workspace_bytes(cfg: Cfg, B: int, T: int) -> int:
    return int(lib().sdm_scan_min_workspace_bytes(ctypes.byref(cfg), B, T))


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A byte tensor of at least nbytes, 256-byte aligned (torch allocations are)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(dev_status: torch.Tensor) -> int:
    """Synchronises (reads the device int) and returns the first device error or 0."""
    return int(dev_status.item())


# ------------------------------------------------------------------ marshalling

def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (there is no CPU path)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(rc: int, what: str):
    if rc != SDM_OK:
        raise SdmError(rc, what)


def _weights(cfg: Cfg, p: Dict[str, torch.Tensor]) -> Weights:
    dt = cfg.torch_dtype
    return Weights(*[_ptr(p[k], dt, k) for k in ("W_qw", "W_qr", "W_v", "K1", "K2")])


def sdm_init_bank(cfg: Cfg, M0: torch.Tensor, banks: torch.Tensor, stream=None) -> None:
    B = banks.shape[0]
    if tuple(banks.shape[1:]) != tuple(M0.shape):
        raise ValueError("banks must be [B, N, d] with M0 [N, d]")
    dt = cfg.torch_dtype
    _check(lib().sdm_init_bank(ctypes.byref(cfg), _ptr(M0, dt, "M0"), _ptr(banks, dt, "banks"),
                               B, _stream(stream)), "sdm_init_bank")


def sdm_project(cfg: Cfg, params: Dict[str, torch.Tensor], x: torch.Tensor, q_w: torch.Tensor,
                q_r: torch.Tensor, v: torch.Tensor, stream=None) -> None:
    dt = cfg.torch_dtype
    ntok = x.numel() // cfg.d
    w = _weights(cfg, params)
    _check(lib().sdm_project(ctypes.byref(cfg), ctypes.byref(w), _ptr(x, dt, "x"), ntok,
                             _ptr(q_w, dt, "q_w"), _ptr(q_r, dt, "q_r"), _ptr(v, dt, "v"),
                             _stream(stream)), "sdm_project")


def sdm_address(cfg: Cfg, K1, K2, q_w, q_r, idx, wsel, ws, dev_status, stream=None) -> None:
    dt = cfg.torch_dtype
    ntok = q_w.numel() // cfg.dk
    _check(lib().sdm_address(ctypes.byref(cfg), _ptr(K1, dt, "K1"), _ptr(K2, dt, "K2"),
                             _ptr(q_w, dt, "q_w"), _ptr(q_r, dt, "q_r"), ntok,
                             _ptr(idx, torch.int32, "idx"), _ptr(wsel, torch.float32, "wsel"),
                             _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                             _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_address")


def sdm_scan(cfg: Cfg, idx, wsel, v, alpha, beta, banks, y, B: int, T: int, ws, dev_status,
             stream=None) -> None:
    dt = cfg.torch_dtype
    _check(lib().sdm_scan(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"),
                          _ptr(wsel, torch.float32, "wsel"), _ptr(v, dt, "v"),
                          _ptr(alpha, torch.float32, "alpha"), _ptr(beta, torch.float32, "beta"),
                          _ptr(banks, dt, "banks"), _ptr(y, torch.float32, "y"), B, T,
                          _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                          _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_scan")


def sdm_scan_prepare(cfg: Cfg, idx, B: int, T: int, ws, dev_status, stream=None) -> None:
    _check(lib().sdm_scan_prepare(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"), B, T,
                                  _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                  _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_scan_prepare")


def sdm_scan_run(cfg: Cfg, idx, wsel, v, alpha, beta, banks, y, B: int, T: int, ws, dev_status,
                 stream=None) -> None:
    dt = cfg.torch_dtype
    _check(lib().sdm_scan_run(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"),
                              _ptr(wsel, torch.float32, "wsel"), _ptr(v, dt, "v"),
                              _ptr(alpha, torch.float32, "alpha"),
                              _ptr(beta, torch.float32, "beta"), _ptr(banks, dt, "banks"),
                              _ptr(y, torch.float32, "y"), B, T, _ptr(ws, None, "ws"),
                              ws.numel() * ws.element_size(),
                              _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_scan_run")


def sdm_scan_run_diag(cfg: Cfg, idx, wsel, v, alpha, beta, banks, y, B: int, T: int, ws,
                      spin_limit_cycles: int, skip_item: int, dev_status, stream=None) -> None:
    """sdm_scan_run with the bound of every wait given in SM clock cycles and, for
    skip_item >= 0, one work item withheld (tests of the failure detection)."""
    dt = cfg.torch_dtype
    _check(lib().sdm_scan_run_diag(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"),
                                   _ptr(wsel, torch.float32, "wsel"), _ptr(v, dt, "v"),
                                   _ptr(alpha, torch.float32, "alpha"),
                                   _ptr(beta, torch.float32, "beta"), _ptr(banks, dt, "banks"),
                                   _ptr(y, torch.float32, "y"), B, T, _ptr(ws, None, "ws"),
                                   ws.numel() * ws.element_size(), int(spin_limit_cycles),
                                   int(skip_item), _ptr(dev_status, torch.int32, "dev_status"),
                                   _stream(stream)),
           "sdm_scan_run_diag")


def sdm_scan_noalloc(cfg: Cfg, idx, wsel, v, alpha, beta, banks, y, B: int, T: int, dev_status,
                     stream=None) -> None:
    """sdm_scan with its scratch in a library-owned device array (no workspace, no
    allocation), for callers that cannot allocate device memory; B * T * w * 4 bytes
    must not exceed SDM_SCAN_NOALLOC_MAX_BYTES (8 MiB)."""
    dt = cfg.torch_dtype
    _check(lib().sdm_scan_noalloc(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"),
                                  _ptr(wsel, torch.float32, "wsel"), _ptr(v, dt, "v"),
                                  _ptr(alpha, torch.float32, "alpha"),
                                  _ptr(beta, torch.float32, "beta"), _ptr(banks, dt, "banks"),
                                  _ptr(y, torch.float32, "y"), B, T,
                                  _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_scan_noalloc")


SCAN_NOALLOC_MAX_BYTES = 8 << 20


def sdm_prefill(cfg: Cfg, params, x, alpha, beta, banks, y, ws, dev_status, idx_out=None,
                w_out=None, stream=None) -> None:
    dt = cfg.torch_dtype
    B, T = x.shape[0], x.shape[1]
    w = _weights(cfg, params)
    _check(lib().sdm_prefill(ctypes.byref(cfg), ctypes.byref(w), _ptr(x, dt, "x"),
                             _ptr(alpha, torch.float32, "alpha"), _ptr(beta, torch.float32, "beta"),
                             _ptr(banks, dt, "banks"), _ptr(y, torch.float32, "y"), B, T,
                             _ptr(idx_out, torch.int32, "idx_out"),
                             _ptr(w_out, torch.float32, "w_out"),
                             _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                             _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_prefill")


def first_touch_bytes(cfg: Cfg, B: int) -> int:
    return int(lib().sdm_first_touch_bytes(ctypes.byref(cfg), B))


def prefill_m0_workspace_bytes(cfg: Cfg, B: int, T: int) -> int:
    return int(lib().sdm_prefill_m0_workspace_bytes(ctypes.byref(cfg), B, T))


def sdm_first_touch(cfg: Cfg, idx, B: int, T: int, first_write, stream=None) -> None:
    _check(lib().sdm_first_touch(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"), B, T,
                                 _ptr(first_write, torch.int32, "first_write"), _stream(stream)),
           "sdm_first_touch")


def sdm_scan_run_m0(cfg: Cfg, idx, wsel, v, alpha, beta, M0, first_write, banks, y, B: int,
                    T: int, ws, dev_status, stream=None) -> None:
    dt = cfg.torch_dtype
    _check(lib().sdm_scan_run_m0(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"),
                                 _ptr(wsel, torch.float32, "wsel"), _ptr(v, dt, "v"),
                                 _ptr(alpha, torch.float32, "alpha"),
                                 _ptr(beta, torch.float32, "beta"), _ptr(M0, dt, "M0"),
                                 _ptr(first_write, torch.int32, "first_write"),
                                 _ptr(banks, dt, "banks"), _ptr(y, torch.float32, "y"), B, T,
                                 _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                 _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_scan_run_m0")


def sdm_fill_untouched(cfg: Cfg, M0, first_write, banks, B: int, T: int, stream=None) -> None:
    dt = cfg.torch_dtype
    _check(lib().sdm_fill_untouched(ctypes.byref(cfg), _ptr(M0, dt, "M0"),
                                    _ptr(first_write, torch.int32, "first_write"),
                                    _ptr(banks, dt, "banks"), B, T, _stream(stream)),
           "sdm_fill_untouched")


def sdm_prefill_m0(cfg: Cfg, params, M0, x, alpha, beta, banks, y, ws, dev_status, idx_out=None,
                   w_out=None, stream=None) -> None:
    """sdm_prefill with banks that start as M0 without a copy (their content on entry is
    ignored); ws: prefill_m0_workspace_bytes(cfg, B, T) bytes."""
    dt = cfg.torch_dtype
    B, T = x.shape[0], x.shape[1]
    w = _weights(cfg, params)
    _check(lib().sdm_prefill_m0(ctypes.byref(cfg), ctypes.byref(w), _ptr(M0, dt, "M0"),
                                _ptr(x, dt, "x"), _ptr(alpha, torch.float32, "alpha"),
                                _ptr(beta, torch.float32, "beta"), _ptr(banks, dt, "banks"),
                                _ptr(y, torch.float32, "y"), B, T,
                                _ptr(idx_out, torch.int32, "idx_out"),
                                _ptr(w_out, torch.float32, "w_out"),
                                _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_prefill_m0")


def tape_bytes(cfg: Cfg, B: int, T: int) -> int:
    return int(lib().sdm_tape_bytes(ctypes.byref(cfg), B, T))


def scan_backward_workspace_bytes(cfg: Cfg, B: int, T: int) -> int:
    return int(lib().sdm_scan_backward_workspace_bytes(ctypes.byref(cfg), B, T))


def sdm_scan_run_train(cfg: Cfg, idx, wsel, v, alpha, beta, banks, y, B: int, T: int, ws, tape,
                       dev_status, M0=None, first_write=None, stream=None) -> None:
    """sdm_scan_run (from M0 when M0 and first_write are given) that also records the
    pre-write values of each token's write slots into tape [B*T, w, d]."""
    dt = cfg.torch_dtype
    _check(lib().sdm_scan_run_train(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"),
                                    _ptr(wsel, torch.float32, "wsel"), _ptr(v, dt, "v"),
                                    _ptr(alpha, torch.float32, "alpha"),
                                    _ptr(beta, torch.float32, "beta"), _ptr(M0, dt, "M0"),
                                    _ptr(first_write, torch.int32, "first_write"),
                                    _ptr(banks, dt, "banks"), _ptr(y, torch.float32, "y"), B, T,
                                    _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                    _ptr(tape, dt, "tape"),
                                    _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_scan_run_train")


def sdm_scan_backward(cfg: Cfg, idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, dalpha,
                      dbeta, dwsel, B: int, T: int, ws, stream=None) -> None:
    """Gradients of the recurrence; banks walk back from the final to the initial state and
    dbank from the final to the initial bank's gradient (see include/sdm.h)."""
    dt = cfg.torch_dtype
    f = torch.float32
    _check(lib().sdm_scan_backward(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"),
                                   _ptr(wsel, f, "wsel"), _ptr(v, dt, "v"),
                                   _ptr(alpha, f, "alpha"), _ptr(beta, f, "beta"),
                                   _ptr(tape, dt, "tape"), _ptr(banks, dt, "banks"),
                                   _ptr(dy, f, "dy"), _ptr(dbank, f, "dbank"), _ptr(dv, f, "dv"),
                                   _ptr(dalpha, f, "dalpha"), _ptr(dbeta, f, "dbeta"),
                                   _ptr(dwsel, f, "dwsel"), B, T, _ptr(ws, None, "ws"),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "sdm_scan_backward")


def address_backward_workspace_bytes(cfg: Cfg, ntok: int) -> int:
    return int(lib().sdm_address_backward_workspace_bytes(ctypes.byref(cfg), ntok))


def sdm_address_backward(cfg: Cfg, K1, K2, q_w, q_r, idx, wsel, dwsel, dq_w, dq_r, dK1, dK2, ws,
                         stream=None) -> None:
    """dq_w, dq_r [ntok, dk] and dK1, dK2 [n, dk/2] (fp32) from the selection-weight
    gradients dwsel [ntok, 2, w], the kept slots idx held fixed."""
    dt = cfg.torch_dtype
    f = torch.float32
    ntok = q_w.shape[0]
    _check(lib().sdm_address_backward(ctypes.byref(cfg), _ptr(K1, dt, "K1"), _ptr(K2, dt, "K2"),
                                      _ptr(q_w, dt, "q_w"), _ptr(q_r, dt, "q_r"), ntok,
                                      _ptr(idx, torch.int32, "idx"), _ptr(wsel, f, "wsel"),
                                      _ptr(dwsel, f, "dwsel"), _ptr(dq_w, f, "dq_w"),
                                      _ptr(dq_r, f, "dq_r"), _ptr(dK1, f, "dK1"), _ptr(dK2, f, "dK2"),
                                      _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                      _stream(stream)),
           "sdm_address_backward")


def project_backward_workspace_bytes(cfg: Cfg, ntok: int) -> int:
    return int(lib().sdm_project_backward_workspace_bytes(ctypes.byref(cfg), ntok))


def sdm_project_backward(cfg: Cfg, params, x, dq_w, dq_r, dv, dx, dW_qw, dW_qr, dW_v, ws,
                         stream=None) -> None:
    """dx [ntok, d], dW_qw, dW_qr [d, dk], dW_v [d, d] (fp32) from the gradients of the
    projection outputs."""
    dt = cfg.torch_dtype
    f = torch.float32
    w = _weights(cfg, params)
    ntok = x.numel() // cfg.d
    _check(lib().sdm_project_backward(ctypes.byref(cfg), ctypes.byref(w), _ptr(x, dt, "x"), ntok,
                                      _ptr(dq_w, f, "dq_w"), _ptr(dq_r, f, "dq_r"), _ptr(dv, f, "dv"),
                                      _ptr(dx, f, "dx"), _ptr(dW_qw, f, "dW_qw"),
                                      _ptr(dW_qr, f, "dW_qr"), _ptr(dW_v, f, "dW_v"),
                                      _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                      _stream(stream)),
           "sdm_project_backward")


def sdm_gdn_dense_scan(cfg: Cfg, kw, kr, k_stride: int, v, alpha, beta, y, B: int, T: int,
                       S0=None, S_out=None, stream=None) -> None:
    """The dense-state comparator: the gated delta rule on a dense [d, 64] fp32 state
    per sequence (kw, kr: fp32 views whose token rows are k_stride floats apart)."""
    for name, t in (("kw", kw), ("kr", kr)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32):
            raise ValueError("%s must be a float32 CUDA tensor (a strided view is fine)" % name)
    _check(lib().sdm_gdn_dense_scan(ctypes.byref(cfg), _ptr(S0, torch.float32, "S0"),
                                    ctypes.c_void_p(kw.data_ptr()), ctypes.c_void_p(kr.data_ptr()),
                                    k_stride, _ptr(v, cfg.torch_dtype, "v"),
                                    _ptr(alpha, torch.float32, "alpha"),
                                    _ptr(beta, torch.float32, "beta"),
                                    _ptr(S_out, torch.float32, "S_out"),
                                    _ptr(y, torch.float32, "y"), B, T, _stream(stream)),
           "sdm_gdn_dense_scan")


def sdm_slot_counts(cfg: Cfg, idx, B: int, T: int, kind: int, t0: int, t1: int, counts,
                    stream=None) -> None:
    """counts [B, N] int32 (uint32 bits) <- per slot, the tokens in [t0, t1) whose write
    (kind 0) or read (kind 1) set holds it."""
    _check(lib().sdm_slot_counts(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"), B, T, kind,
                                 t0, t1, _ptr(counts, torch.int32, "counts"), _stream(stream)),
           "sdm_slot_counts")


def slot_overlap_workspace_bytes(cfg: Cfg, B: int) -> int:
    return int(lib().sdm_slot_overlap_workspace_bytes(ctypes.byref(cfg), B))


def sdm_slot_overlap(cfg: Cfg, idx, B: int, T: int, w0: int, w1: int, r0: int, r1: int, out, ws,
                     stream=None) -> None:
    """out [B, 3] int32 <- distinct slots written in [w0, w1), read in [r0, r1), and in both."""
    _check(lib().sdm_slot_overlap(ctypes.byref(cfg), _ptr(idx, torch.int32, "idx"), B, T, w0, w1,
                                  r0, r1, _ptr(out, torch.int32, "out"), _ptr(ws, None, "ws"),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "sdm_slot_overlap")


def sdm_decode_step(cfg: Cfg, params, x, alpha, beta, banks, y, ws, dev_status,
                    idx_out=None, w_out=None, stream=None) -> None:
    """One token for each of B sequences; idx_out / w_out [B, 2, w] optionally receive
    the slot sets and weights the step used."""
    dt = cfg.torch_dtype
    B = x.shape[0]
    w = _weights(cfg, params)
    _check(lib().sdm_decode_step(ctypes.byref(cfg), ctypes.byref(w), _ptr(x, dt, "x"),
                                 _ptr(alpha, torch.float32, "alpha"),
                                 _ptr(beta, torch.float32, "beta"), _ptr(banks, dt, "banks"),
                                 _ptr(y, torch.float32, "y"), B,
                                 _ptr(idx_out, torch.int32, "idx_out"),
                                 _ptr(w_out, torch.float32, "w_out"), _ptr(ws, None, "ws"),
                                 ws.numel() * ws.element_size(),
                                 _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
           "sdm_decode_step")
