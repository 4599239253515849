"""Seeded synthetic inputs for Sparse Delta Memory (SDM) layer workloads.

This module is shared by the CPU oracle tests and by the CUDA path (tests, the
smoke check and the benchmark). It holds no arithmetic of the method: it only
draws random tensors with the shapes and distributions of the workloads and
returns them as CPU torch tensors. Both sides receive the same bits.

Distributions (one Sparse Delta Memory layer; the pages give N = 480^2 slots and
W = 64 active slots, blog "Background"; d = 3840 for the 8B illustration, blog
"Unlocking linear memory states through sparsity"):

- x ~ N(0, 1); W_qw, W_qr, W_v ~ N(0, std 1/sqrt(d)); K1, K2 ~ N(0, std 1/sqrt(dk/2));
- M0 ~ N(0, std 0.02) (one learned initial state shared by all sequences);
- alpha = sigmoid(g + 3), beta = sigmoid(b) with g, b ~ N(0, 1), per token.

Every tensor has its own torch.Generator seeded with seed * 100 + tensor_id and is
drawn in fp32, then cast (round-to-nearest-even) to bf16 where the workload is bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

# tensor ids (each tensor gets its own generator stream)
_X, _WQW, _WQR, _WV, _K1, _K2, _M0, _G, _BB = 1, 2, 3, 4, 5, 6, 7, 8, 9
_POOL, _POOL_MASK, _POOL_PICK_W, _POOL_PICK_R = 10, 11, 12, 13
_PAT_Q, _PAT_V = 14, 15
_DEC_X, _DEC_G, _DEC_B = 16, 17, 18


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and structure of one synthetic SDM workload."""

    name: str
    B: int            # sequences
    T: int            # tokens per sequence (prefill); for decode: prior writes
    d: int            # slot width / model width
    n: int            # sub-key rows; N = n * n slots
    dk: int           # query width (dk / 2 per half)
    W: int            # active slots per token (write and read)
    dtype: str        # "f32" or "bf16": storage of x, weights, keys, banks, q, v
    seed: int
    pool_frac: float = 0.0      # fraction of tokens whose q^w, q^r come from a pool
    pool_size: int = 0
    pattern_len: int = 0        # tokens of an inserted key/value pattern
    pattern_write_at: int = 0
    pattern_read_at: int = 0
    decode_steps: int = 0       # decode workloads: steps after the T prior writes

    @property
    def N(self) -> int:
        return self.n * self.n

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the benchmark spec, named by what they are.
WORKLOADS: Dict[str, Workload] = {
    "tiny-f32": Workload("tiny-f32", B=1, T=256, d=64, n=32, dk=64, W=8,
                         dtype="f32", seed=1001),
    "prefill-d2048-b4": Workload("prefill-d2048-b4", B=4, T=4096, d=2048, n=480,
                                 dk=256, W=64, dtype="bf16", seed=1002),
    "decode-d2048-b64": Workload("decode-d2048-b64", B=64, T=1024, d=2048, n=480,
                                 dk=256, W=64, dtype="bf16", seed=1003,
                                 decode_steps=512),
    "prefill-d3840-pool": Workload("prefill-d3840-pool", B=2, T=16384, d=3840, n=480,
                                   dk=256, W=64, dtype="bf16", seed=1004,
                                   pool_frac=0.3, pool_size=64),
    "long-131k": Workload("long-131k", B=1, T=131072, d=2048, n=480, dk=256, W=64,
                          dtype="bf16", seed=1005, pattern_len=16,
                          pattern_write_at=8000, pattern_read_at=130000),
}


def _gen(wl: Workload, tid: int) -> torch.Generator:
    return torch.Generator().manual_seed(wl.seed * 100 + tid)


def _randn(wl: Workload, tid: int, shape, std: float = 1.0, mean: float = 0.0) -> torch.Tensor:
    t = torch.randn(*shape, generator=_gen(wl, tid), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def _cast(wl: Workload, t: torch.Tensor) -> torch.Tensor:
    return t if wl.dtype == "f32" else t.to(torch.bfloat16)


def _gates(wl: Workload, tid_g: int, tid_b: int, shape):
    alpha = torch.sigmoid(_randn(wl, tid_g, shape) + 3.0)
    beta = torch.sigmoid(_randn(wl, tid_b, shape))
    return alpha.contiguous(), beta.contiguous()


def make_params(wl: Workload, with_m0: bool = True) -> Dict[str, torch.Tensor]:
    """Layer parameters: projections, sub-key tables and the initial state M0."""
    d, dk, n = wl.d, wl.dk, wl.n
    p = {
        "W_qw": _cast(wl, _randn(wl, _WQW, (d, dk), 1.0 / math.sqrt(d))),
        "W_qr": _cast(wl, _randn(wl, _WQR, (d, dk), 1.0 / math.sqrt(d))),
        "W_v": _cast(wl, _randn(wl, _WV, (d, d), 1.0 / math.sqrt(d))),
        "K1": _cast(wl, _randn(wl, _K1, (n, dk // 2), 1.0 / math.sqrt(dk // 2))),
        "K2": _cast(wl, _randn(wl, _K2, (n, dk // 2), 1.0 / math.sqrt(dk // 2))),
    }
    if with_m0:
        p["M0"] = _cast(wl, _randn(wl, _M0, (wl.N, d), 0.02))
    return p


def make_tokens(wl: Workload) -> Dict[str, torch.Tensor]:
    """Per-token inputs of a prefill: x [B,T,d], alpha [B,T], beta [B,T] (fp32)."""
    x = _cast(wl, _randn(wl, _X, (wl.B, wl.T, wl.d)))
    alpha, beta = _gates(wl, _G, _BB, (wl.B, wl.T))
    return {"x": x, "alpha": alpha, "beta": beta}


def make_decode_tokens(wl: Workload) -> Dict[str, torch.Tensor]:
    """Decode inputs: x [steps,B,d], alpha/beta [steps,B] for `decode_steps` steps."""
    s = wl.decode_steps
    x = _cast(wl, _randn(wl, _DEC_X, (s, wl.B, wl.d)))
    alpha, beta = _gates(wl, _DEC_G, _DEC_B, (s, wl.B))
    return {"x": x, "alpha": alpha, "beta": beta}


def make_pool(wl: Workload) -> Optional[Dict[str, torch.Tensor]]:
    """Query pool: each token independently (prob pool_frac) takes its q^w and q^r
    from a pool of `pool_size` vectors ~N(0,1); the pool entries for q^w and q^r
    are picked independently. Returns mask [B,T] bool, pick_w/pick_r [B,T] int64,
    pool [pool_size, dk] (I/O dtype)."""
    if wl.pool_frac <= 0.0:
        return None
    pool = _cast(wl, _randn(wl, _POOL, (wl.pool_size, wl.dk)))
    mask = torch.rand(wl.B, wl.T, generator=_gen(wl, _POOL_MASK)) < wl.pool_frac
    pick_w = torch.randint(0, wl.pool_size, (wl.B, wl.T), generator=_gen(wl, _POOL_PICK_W))
    pick_r = torch.randint(0, wl.pool_size, (wl.B, wl.T), generator=_gen(wl, _POOL_PICK_R))
    return {"pool": pool, "mask": mask, "pick_w": pick_w, "pick_r": pick_r}


def make_pattern(wl: Workload) -> Optional[Dict[str, torch.Tensor]]:
    """Inserted key/value pattern: for i < pattern_len, token write_at+i writes with
    q^w := p_i and v := v_i; token read_at+i reads with q^r := p_i.
    Returns p [L, dk] and v [L, d] (I/O dtype) and the two positions."""
    if wl.pattern_len <= 0:
        return None
    p = _cast(wl, _randn(wl, _PAT_Q, (wl.pattern_len, wl.dk)))
    v = _cast(wl, _randn(wl, _PAT_V, (wl.pattern_len, wl.d)))
    return {"p": p, "v": v,
            "write_at": torch.tensor(wl.pattern_write_at),
            "read_at": torch.tensor(wl.pattern_read_at)}


def inject_queries(wl: Workload, q_w: torch.Tensor, q_r: torch.Tensor, v: torch.Tensor,
                   pool=None, pattern=None) -> None:
    """Overwrite projected q^w, q^r [B,T,dk] and v [B,T,d] in place with the pool or
    pattern vectors of the workload (a data substitution, no arithmetic). Works on
    CPU or device tensors."""
    if pool is not None:
        m = pool["mask"].to(q_w.device)
        pw = pool["pool"].to(q_w.device)[pool["pick_w"].to(q_w.device)]
        pr = pool["pool"].to(q_w.device)[pool["pick_r"].to(q_w.device)]
        q_w[m] = pw[m]
        q_r[m] = pr[m]
    if pattern is not None:
        L = pattern["p"].shape[0]
        wa, ra = int(pattern["write_at"]), int(pattern["read_at"])
        p = pattern["p"].to(q_w.device)
        q_w[:, wa:wa + L] = p
        v[:, wa:wa + L] = pattern["v"].to(v.device)
        q_r[:, ra:ra + L] = p
