"""GB300-native fused attention for large head dimensions (D = 64..1024).

The computation runs in libffpa.so (hand-written sm_103a kernels behind a C
ABI, declared in include/ffpa.h).  This package only builds and loads that
library and marshals torch tensors into its descriptors; PyTorch supplies
device memory and streams.

    from head_dim_attention_gb300 import attention_fwd, attention_bwd
    out, lse = attention_fwd(q, k, v, causal=True)
    dq, dk, dv = attention_bwd(q, k, v, out, lse, dout, causal=True)
"""
from __future__ import annotations

import math

from ._lib import (  # noqa: F401
    FfpaError,
    ffpa_bwd,
    ffpa_bwd_dropout,
    ffpa_check_status,
    ffpa_fwd,
    ffpa_fwd_dropout,
    ffpa_status_string,
    ffpa_version,
    load,
)

__all__ = ["attention_fwd", "attention_bwd", "ffpa_fwd", "ffpa_bwd", "ffpa_fwd_dropout", "ffpa_bwd_dropout",
           "ffpa_check_status",
           "ffpa_status_string", "ffpa_version", "FfpaError", "load"]


def attention_fwd(q, k, v, bias=None, causal=False, scale=None, out=None, lse=None, stream=None,
                  dropout_p=0.0, seed=0, offset=0):
    """O and lse for q [B,Hq,Nq,D], k/v [B,Hkv,Nkv,D] (CUDA f16/bf16); allocates out/lse if not given.

    dropout_p > 0 drops attention probabilities under the library's Philox
    contract (include/ffpa.h, ffpa_fwd_dropout) with the given seed and offset.
    """
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if dropout_p:
        ffpa_fwd_dropout(q, k, v, bias, causal, scale, dropout_p, seed, offset, out, lse, stream)
    else:
        ffpa_fwd(q, k, v, bias, causal, scale, out, lse, stream)
    return out, lse


def attention_bwd(q, k, v, out, lse, dout, bias=None, causal=False, scale=None, dq=None, dk=None, dv=None,
                  stream=None, dropout_p=0.0, seed=0, offset=0):
    """dQ, dK, dV for the forward that produced ``out`` and ``lse`` (with the same
    dropout_p, seed and offset); allocates outputs if not given."""
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dropout_p:
        ffpa_bwd_dropout(q, k, v, bias, causal, scale, dropout_p, seed, offset, out, lse, dout, dq, dk, dv, stream)
    else:
        ffpa_bwd(q, k, v, bias, causal, scale, out, lse, dout, dq, dk, dv, stream)
    return dq, dk, dv
