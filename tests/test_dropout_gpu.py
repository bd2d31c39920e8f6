"""Dropout on the attention probabilities: the C-ABI path against the oracle.

Both sides draw the keep mask from the same Philox4x32-10 contract
(include/ffpa.h, ffpa_fwd_dropout); the oracle's generator is pinned against
the published known-answer vectors (tests/test_oracle.py).  The mask decides
an integer (kept or not), so it is checked bit-exactly through a
construction that makes O and dV show it directly; O, lse and the gradients
are then checked at the usual tolerances on small shapes (every kernel
flavour: D <= 512 and D > 512, causal, GQA, bias, ragged tails) and on the
workload-sized case by sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle.attn_ref as ref
from head_dim_attention_gb300 import (FfpaError, attention_bwd, attention_fwd, ffpa_check_status,
                                      ffpa_fwd_dropout)
from parity import check_bwd_full, check_bwd_sampled, check_fwd_full, check_fwd_sampled

pytestmark = pytest.mark.gpu
BF, FP = torch.bfloat16, torch.float16


@pytest.mark.parametrize("D,Nkv,Nq,p", [(512, 512, 300, 0.3), (1024, 640, 200, 0.5), (320, 256, 129, 0.1)])
def test_keep_mask_bit_exact(D, Nkv, Nq, p):
    # Q = 0 makes every probability 1 / Nkv; V = [I 0] and dO = [I 0] make
    # O[i, j] = keep_ij / ((1 - p) Nkv) and dV[j, i] = keep_ij / ((1 - p) Nkv):
    # the kept scores are exactly the positive entries
    B, Hq, Hkv = 2, 2, 1
    seed, offset = 0x5EED0123456789AB, 17
    dev = torch.device("cuda")
    q = torch.zeros(B, Hq, Nq, D, dtype=BF, device=dev)
    k = torch.randn(B, Hkv, Nkv, D, device=dev).to(BF)
    v = torch.zeros(B, Hkv, Nkv, D, dtype=BF, device=dev)
    v[..., :, :Nkv] = torch.eye(Nkv, dtype=BF, device=dev)  # Nkv <= D
    do = torch.zeros(B, Hq, Nq, D, dtype=BF, device=dev)
    do[..., :, :Nq] = torch.eye(Nq, dtype=BF, device=dev)
    out, lse = attention_fwd(q, k, v, dropout_p=p, seed=seed, offset=offset)
    dq, dk, dv = attention_bwd(q, k, v, out, lse, do, dropout_p=p, seed=seed, offset=offset)
    torch.cuda.synchronize()
    assert ffpa_check_status() == 0
    o = out.float().cpu().numpy()
    dvn = dv.float().cpu().numpy()
    group = Hq // Hkv
    for b in range(B):
        kv_sum = np.zeros((Nkv, Nq))
        for h in range(Hq):
            keep = ref.dropout_keep(b, h, Hq, np.arange(Nq), np.arange(Nkv), p, seed, offset)
            assert np.array_equal(o[b, h, :, :Nkv] > 0, keep), (b, h, int(np.sum((o[b, h, :, :Nkv] > 0) != keep)))
            assert np.all(o[b, h, :, Nkv:] == 0)
            kv_sum += keep.T
        # dV sums the group's query heads: the count of heads that keep (i, j)
        want = kv_sum / ((1.0 - p) * Nkv)
        got = dvn[b, 0, :, :Nq]
        assert np.allclose(got, want, rtol=1e-2, atol=1e-6), (b, float(np.max(np.abs(got - want))))
        assert np.array_equal(got > 0, kv_sum > 0)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,dtype,causal,bias", [
    (1, 2, 1, 300, 333, 512, BF, False, True),
    (1, 2, 2, 129, 129, 512, FP, True, False),
    (2, 2, 1, 200, 140, 384, BF, True, True),
    (1, 4, 2, 17, 260, 640, BF, False, False),
    (1, 2, 1, 256, 300, 1024, FP, True, True),
    (1, 1, 1, 5, 200, 832, BF, False, False),
    (1, 4, 2, 200, 300, 768, BF, True, True),
    (2, 4, 1, 130, 260, 448, FP, True, False),
])
def test_dropout_fwd_bwd_small(B, Hq, Hkv, Nq, Nkv, D, dtype, causal, bias):
    drop = (0.2, 0xC0FFEE, 3)
    check_fwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=causal, bias=bias, dropout=drop)
    check_bwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=causal, bias=bias, dropout=drop)


def test_dropout_8k_bf16_sampled():
    # the workload-sized configuration with dropout, on 64 seeded rows per head
    drop = (0.1, 1234567, 0)
    check_fwd_sampled(1, 8, 8, 8192, 8192, 512, BF, dropout=drop)
    check_bwd_sampled(1, 8, 8, 8192, 8192, 512, BF, dropout=drop)


def test_dropout_p0_and_rejections():
    dev = torch.device("cuda")
    q = torch.randn(1, 2, 130, 512, device=dev).to(BF)
    k = torch.randn(1, 2, 140, 512, device=dev).to(BF)
    v = torch.randn(1, 2, 140, 512, device=dev).to(BF)
    o0, l0 = attention_fwd(q, k, v)
    o1, l1 = torch.empty_like(o0), torch.empty_like(l0)
    ffpa_fwd_dropout(q, k, v, None, 0, 512 ** -0.5, 0.0, 5, 0, o1, l1)  # p = 0: the call without dropout
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    for bad in (1.0, -0.1, float("nan")):
        with pytest.raises(FfpaError):
            attention_fwd(q, k, v, dropout_p=bad, seed=1)
    small = torch.randn(1, 2, 130, 128, device=dev).to(BF)
    with pytest.raises(FfpaError):
        attention_fwd(small, small, small, dropout_p=0.1, seed=1)
