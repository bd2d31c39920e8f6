"""Backward parity: dQ/dK/dV from the C-ABI path against the fp64 oracle.

The bar is a relative Frobenius error <= 2e-2 per gradient tensor.  Small
shapes are checked over the whole tensors (tails, GQA, bias, causal with
Nq != Nkv, every head-dimension regime); the workload-sized self-attention
case (B=1, H=8, N=8192, D=512, bf16, causal and not) is checked on 64 seeded
query rows and 64 seeded key rows per head, with the oracle computing the
full-row statistics it needs itself.
"""
import pytest
import torch

from parity import check_bwd_full, check_bwd_sampled

pytestmark = pytest.mark.gpu
BF, FP = torch.bfloat16, torch.float16


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,dtype,causal,bias", [
    (1, 1, 1, 256, 256, 512, FP, False, False),
    (1, 2, 2, 129, 129, 512, BF, True, False),
    (1, 4, 2, 200, 333, 512, FP, False, True),
    (2, 2, 1, 255, 255, 320, BF, True, True),
    (1, 1, 1, 130, 130, 256, BF, False, False),
    (1, 1, 1, 64, 64, 64, FP, False, False),
    (1, 2, 1, 300, 100, 576, BF, True, False),
    (1, 1, 1, 100, 300, 1024, FP, True, False),
    (1, 1, 1, 17, 140, 768, BF, False, True),
    (1, 2, 2, 5, 200, 512, BF, False, False),
    (1, 4, 1, 384, 384, 640, FP, True, True),
    # D = 512 runs as CTA pairs over neighbouring stationary tiles: odd tile
    # counts (the last pair's second tile is empty), causal with Nq != Nkv,
    # GQA with bias, a single query row
    (1, 4, 2, 300, 500, 512, BF, True, True),
    (1, 2, 1, 500, 300, 512, FP, True, False),
    (2, 2, 2, 384, 384, 512, BF, False, False),
    (1, 1, 1, 1, 129, 512, BF, False, False),
    # the same pair kernels at D = 320 .. 448 (odd chunk counts pad the last
    # gradient quarter; dV's second half is 128 or 256 columns wide)
    (1, 4, 2, 300, 500, 384, BF, True, True),
    (1, 2, 1, 500, 300, 448, FP, True, False),
    (2, 2, 2, 384, 384, 448, BF, False, False),
    (1, 2, 2, 200, 333, 320, FP, False, True),
    (1, 2, 2, 5, 200, 384, BF, False, False),
    # D = 576 .. 1024: the exchange kernel's two modes (two ranges of gradient
    # columns; a range that is not a multiple of 128 pads with zero-filled
    # operand columns), with tails, GQA, bias and causal
    (1, 4, 2, 300, 500, 832, BF, True, True),
    (1, 2, 1, 260, 130, 960, FP, False, False),
    (2, 2, 2, 256, 256, 704, BF, True, False),
    (1, 2, 2, 5, 200, 896, BF, False, True),
    (1, 2, 1, 129, 383, 1024, BF, False, True),
])
def test_bwd_small(B, Hq, Hkv, Nq, Nkv, D, dtype, causal, bias):
    check_bwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=causal, bias=bias)


def test_bwd_query_bias_small():
    check_bwd_full(1, 2, 2, 150, 260, 512, BF, bias="query")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_8k_bf16(causal):
    check_bwd_sampled(1, 8, 8, 8192, 8192, 512, BF, causal=causal)


@pytest.mark.parametrize("D", [320, 384, 448, 640, 832, 1024])
def test_bwd_4k_head_dims(D):
    check_bwd_sampled(1, 4, 4, 4096, 4096, D, FP, causal=(D in (384, 832)))
