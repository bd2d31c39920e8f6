"""The decode forward without allocation, against the ordinary decode path.

ffpa_fwd_decode_noalloc serves callers that cannot allocate device memory
during the call (code running under another framework's memory pool, or a
serving loop that must stay out of the CUDA allocator).  It runs the same
decode kernels as ffpa_fwd but keeps the per-slice partials in a fixed device
array inside the library.  This test calls it through the C ABI twice in a
row (the array keeps the previous call's contents, so the second call checks
that nothing stale leaks in) and compares each result with ffpa_fwd's, within
the forward parity tolerance.  It also checks that a call needing more than
the fixed scratch is refused without launching anything.  The file is named
to be collected last.
"""
import numpy as np
import pytest
import torch

from head_dim_attention_gb300 import _lib, ffpa_check_status
from head_dim_attention_gb300.synth import make_inputs
from parity import LSE_ATOL, TOL, assert_close

pytestmark = pytest.mark.gpu


def _run(fn, inp, causal, scale):
    dev = torch.device("cuda")
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    bias = None if inp.bias is None else inp.bias.to(dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    fn(q, k, v, bias, causal, scale, out, lse)
    torch.cuda.synchronize()
    assert ffpa_check_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,dtype,causal,bias", [
    (1, 8, 8, 1, 8192, 512, torch.bfloat16, False, False),
    (1, 4, 2, 3, 1000, 320, torch.float16, True, True),
])
def test_noalloc_matches_decode_path_twice(B, Hq, Hkv, Nq, Nkv, D, dtype, causal, bias):
    scale = D ** -0.5
    atol, rtol = TOL[dtype]
    for seed in (0, 1):  # two calls in a row on different inputs
        inp = make_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, bias=bias, seed=seed)
        o_ref, l_ref = _run(_lib.ffpa_fwd, inp, causal, scale)
        o_new, l_new = _run(_lib.ffpa_fwd_decode_noalloc, inp, causal, scale)
        assert np.isfinite(o_new).all() and np.isfinite(l_new).all()
        assert_close(o_new, o_ref, atol, rtol, f"O (call {seed + 1})")
        assert_close(l_new, l_ref, LSE_ATOL, 0.0, f"lse (call {seed + 1})")


def test_noalloc_refuses_oversized_call():
    # B=8, Hq=8, Nq=16, Nkv=2048, D=1024: slices hold at most 256 keys, so at least
    # 8*8*16*8 slice rows * 1026 floats (33.6 MB) > 8 MiB
    dev = torch.device("cuda")
    q = torch.zeros(8, 8, 16, 1024, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(8, 8, 2048, 1024, dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    with pytest.raises(_lib.FfpaError) as err:
        _lib.ffpa_fwd_decode_noalloc(q, k, k, None, 0, 0.03, out, None)
    assert err.value.code == 6
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0  # nothing was launched
