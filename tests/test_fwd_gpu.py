"""Forward parity: the C-ABI CUDA path against the fp64 oracle on seeded inputs.

Small shapes are compared element by element over the whole output; they span
several 128-row tiles, ragged tails, both dtypes, every head-dimension regime
of the fused kernels (one CTA for D <= 256; a CTA pair holding all of O for
D = 320..512; two pairs splitting O along D at D = 576 and 640 and with
dropout or key splits above; a score pair and an O pair for D = 704..1024)
and the decode path (Nq <= 16).  The workload-sized cases compare 64 seeded
query rows per head, which the oracle computes one by one.
"""
import pytest
import torch

from parity import check_fwd_full, check_fwd_sampled

pytestmark = pytest.mark.gpu
BF, FP = torch.bfloat16, torch.float16


def test_config_small_self_attention():
    # B=1, H=1, N=256, D=512, fp16, scale 1/sqrt(512), seed 0: full output
    check_fwd_full(1, 1, 1, 256, 256, 512, FP)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,dtype,causal,bias", [
    (1, 2, 2, 129, 129, 512, BF, False, False),
    (1, 2, 2, 200, 333, 512, BF, False, True),
    (1, 4, 1, 300, 300, 512, FP, True, False),
    (2, 2, 1, 255, 255, 320, BF, True, True),
    (1, 1, 1, 128, 1000, 576, FP, False, False),
    (1, 1, 1, 257, 384, 1024, BF, True, False),
    (1, 2, 2, 130, 130, 256, BF, False, False),
    (1, 1, 1, 64, 64, 64, FP, False, False),
    (1, 2, 2, 17, 140, 768, BF, False, True),
    (1, 1, 1, 300, 100, 512, BF, True, False),
    (1, 1, 1, 100, 300, 512, FP, True, True),
    (1, 2, 1, 384, 384, 640, FP, False, False),
    (1, 1, 1, 127, 1, 448, BF, False, False),
    # GQA + key bias + causal + ragged at D=512 (early rows see few keys, so
    # outputs can be sums of nearly cancelling V rows)
    (1, 2, 1, 200, 200, 512, BF, True, True),
    (1, 2, 2, 200, 200, 512, BF, True, True),
    (1, 4, 2, 333, 333, 512, FP, True, True),
    # the same at the other full-D pair widths (O's second half N = 128 or 256)
    (1, 4, 2, 333, 333, 384, BF, True, True),
    (1, 2, 1, 200, 300, 448, FP, False, True),
    (2, 2, 2, 190, 190, 320, FP, True, False),
    # the score pair + O pair kernel (D >= 704) with GQA, two batches, causal
    # with Nq != Nkv and a key bias
    (2, 4, 2, 200, 300, 1024, BF, True, True),
    (1, 4, 1, 300, 200, 832, FP, False, False),
])
def test_fused_small(B, Hq, Hkv, Nq, Nkv, D, dtype, causal, bias):
    check_fwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=causal, bias=bias)


@pytest.mark.parametrize("sharp,dtype", [(1.5, BF), (2.0, BF), (3.0, BF), (2.0, FP), (6.0, FP)])
def test_sharp_softmax(sharp, dtype):
    # Scores with standard deviation `sharp`: from rows whose weight is spread
    # over many keys to rows that a few keys dominate, so key tiles that feed P
    # as one 16-bit term and tiles that add its rounding residual mix within a
    # row and within a tile.
    check_fwd_full(1, 2, 2, 700, 1100, 512, dtype, scale=sharp * 512 ** -0.5)


@pytest.mark.parametrize("D", [320, 384, 448, 640, 768, 1024])
def test_sharp_softmax_head_dims(D):
    check_fwd_full(1, 2, 2, 700, 1100, D, BF, scale=2.0 * D ** -0.5)


def test_sharp_softmax_8k_bf16():
    check_fwd_sampled(1, 2, 2, 8192, 8192, 512, BF, scale=2.0 * 512 ** -0.5)


def test_fused_query_bias_small():
    # [1, 1, Nq, Nkv] per-query bias
    check_fwd_full(1, 2, 2, 150, 260, 512, torch.bfloat16, bias="query")


@pytest.mark.parametrize("D", [320, 384, 448, 512, 576, 640, 704, 768, 832, 896, 960, 1024])
def test_head_dim_sweep_small(D):
    check_fwd_full(1, 2, 2, 200, 200, D, FP, causal=(D % 128 == 0))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,dtype,causal,bias", [
    (1, 8, 8, 1, 1000, 512, BF, False, False),
    (1, 4, 2, 3, 257, 512, FP, True, True),
    (2, 2, 2, 16, 130, 1024, BF, False, False),
    (1, 2, 1, 5, 1, 320, FP, False, True),
    (1, 1, 1, 16, 16, 64, BF, True, False),
    # one or two query rows with contiguous K/V rows stream the slice through
    # shared memory: GQA + bias + causal, head dimensions whose 16-byte groups
    # do not fill every lane, ragged slices, a slice of a single partial stage
    (1, 4, 2, 2, 1000, 512, BF, True, True),
    (2, 3, 3, 1, 777, 320, FP, False, True),
    (1, 2, 1, 2, 8191, 448, BF, False, False),
    (1, 1, 1, 1, 17, 512, FP, True, False),
    # a CTA takes the whole GQA group when group x Nq <= 4 (D <= 512) or <= 2:
    # groups of 4 and 3, D > 512 with a group of 2, and a group of 4 that
    # does not fit at D > 512
    (1, 8, 2, 1, 1500, 512, BF, False, True),
    (1, 6, 2, 1, 333, 320, FP, True, True),
    (1, 4, 2, 1, 500, 1024, FP, True, False),
    (2, 4, 1, 1, 700, 768, BF, False, True),
])
def test_decode_small(B, Hq, Hkv, Nq, Nkv, D, dtype, causal, bias):
    check_fwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=causal, bias=bias)


# ---------------------------------------------------------------- workload-sized cases
def test_self_attention_8k_bf16():
    check_fwd_sampled(1, 8, 8, 8192, 8192, 512, BF)


@pytest.mark.parametrize("D", [320, 384, 448, 512, 576, 640, 768, 1024])
def test_head_dim_sweep_4k_fp16(D):
    check_fwd_sampled(1, 8, 8, 4096, 4096, D, FP)


def test_causal_8k():
    check_fwd_sampled(1, 8, 8, 8192, 8192, 512, BF, causal=True)


def test_gqa_8k():
    check_fwd_sampled(1, 8, 2, 8192, 8192, 512, BF)


def test_non_aligned_8191():
    check_fwd_sampled(1, 8, 8, 8191, 8191, 512, BF)


def test_cross_attention_bias():
    check_fwd_sampled(1, 8, 8, 1024, 8192, 512, BF, bias=True)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,dtype,causal,bias", [
    (1, 8, 2, 64, 8192, 512, BF, False, True),
    (1, 4, 4, 17, 3000, 384, FP, True, False),   # causal: the later key splits see no key
    (2, 2, 1, 40, 5000, 1024, BF, False, False),  # O split over pairs and keys split
    (1, 1, 1, 130, 2048, 576, FP, True, True),
])
def test_short_query_key_splits(B, Hq, Hkv, Nq, Nkv, D, dtype, causal, bias):
    # 17..130 query rows fill a fraction of a wave of CTA pairs: the keys are
    # split between pairs and the partials merged by the decode combine
    check_fwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=causal, bias=bias)


def test_decode_8k():
    check_fwd_full(1, 8, 8, 1, 8192, 512, BF)


def test_decode_gqa_8k():
    # Hq = 8 on Hkv = 2: one CTA per (slice, kv head) scores all four query heads
    check_fwd_full(1, 8, 2, 1, 8192, 512, BF)


@pytest.mark.parametrize("Hq,Hkv,Nq,D", [(8, 2, 1, 512), (4, 2, 2, 448), (2, 2, 2, 768), (4, 4, 3, 512)])
def test_decode_strided_kv_rows(Hq, Hkv, Nq, D):
    # K and V rows D + 64 elements apart: the register-fed kernel instead of
    # the shared-memory one, with and without a shared GQA group
    check_fwd_full(1, Hq, Hkv, Nq, 900, D, BF, causal=True, bias=True, kv_row_pad=64)
