"""Helpers for the GPU parity tests: run the C-ABI path, run the oracle, compare.

Tolerances are the ones the task fixes for this method:
  O:    |gpu - ref| <= 2e-3 + 2e-2 |ref| (bf16),  1e-3 + 5e-3 |ref| (fp16)
  lse:  |gpu - ref| <= 1e-3
  dQ/dK/dV: relative Frobenius error ||gpu - ref||_F / ||ref||_F <= 2e-2, per
            tensor and, where whole tensors are compared, also per 128-row
            tile of every (batch, head), so one wrong tile (a ragged tail, a
            causal diagonal block) cannot hide under the whole tensor's norm;
            a tile whose exact gradient is zero (keys no query sees) must come
            back zero
With dropout (``dropout=(p, seed, offset)``) both sides draw the keep mask
from the same Philox contract; the same tolerances apply.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.attn_ref as ref
from head_dim_attention_gb300 import attention_bwd, attention_fwd, ffpa_check_status
from head_dim_attention_gb300.synth import make_inputs

TOL = {torch.bfloat16: (2e-3, 2e-2), torch.float16: (1e-3, 5e-3)}
LSE_ATOL = 1e-3
GRAD_RTOL = 2e-2


def f64(t):
    return None if t is None else t.double().numpy()


def assert_close(gpu, want, atol, rtol, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert gpu.shape == want.shape, (what, gpu.shape, want.shape)
    same_inf = np.isinf(want) & (gpu == want)
    err = np.where(same_inf, 0.0, np.abs(gpu - want))
    bound = atol + rtol * np.where(np.isinf(want), 0.0, np.abs(want))
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={gpu[i]!r} ref={want[i]!r}")


def rel_fro(gpu, want):
    gpu = np.asarray(gpu, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(gpu - want) / max(np.linalg.norm(want), 1e-300))


def tile_errors(gpu, want, what, tile=128):
    """Relative Frobenius error of every `tile`-row block of every (batch, head) of a gradient."""
    gpu = np.asarray(gpu, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    errs = {}
    for b in range(want.shape[0]):
        for h in range(want.shape[1]):
            for r0 in range(0, want.shape[2], tile):
                g, w = gpu[b, h, r0:r0 + tile], want[b, h, r0:r0 + tile]
                key = f"{what}[b={b},h={h},rows {r0}..{r0 + len(w) - 1}]"
                nw = np.linalg.norm(w)
                errs[key] = float(np.linalg.norm(g - w) / nw) if nw > 0 else (0.0 if not np.any(g) else np.inf)
    return errs


def _row_padded(t, pad, dev):
    """The same values in a buffer whose rows are `pad` elements longer (a
    non-contiguous row stride, as a slice of a wider tensor would have)."""
    if not pad:
        return t.to(dev)
    wide = torch.zeros(*t.shape[:-1], t.shape[-1] + pad, dtype=t.dtype, device=dev)
    wide[..., : t.shape[-1]] = t.to(dev)
    return wide[..., : t.shape[-1]]


def _drop_kw(dropout):
    if dropout is None:
        return {}
    p, seed, offset = dropout
    return {"dropout_p": p, "seed": seed, "offset": offset}


def gpu_fwd(inp, causal, scale, kv_row_pad=0, dropout=None):
    dev = torch.device("cuda")
    q = inp.q.to(dev)
    k, v = _row_padded(inp.k, kv_row_pad, dev), _row_padded(inp.v, kv_row_pad, dev)
    bias = None if inp.bias is None else inp.bias.to(dev)
    out, lse = attention_fwd(q, k, v, bias=bias, causal=causal, scale=scale, **_drop_kw(dropout))
    torch.cuda.synchronize()
    assert ffpa_check_status() == 0
    return out, lse


def check_fwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=False, bias=False, seed=0, scale=None, kv_row_pad=0,
                   dropout=None):
    inp = make_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, bias=bias, seed=seed)
    scale = D ** -0.5 if scale is None else scale
    out, lse = gpu_fwd(inp, causal, scale, kv_row_pad, dropout=dropout)
    o_ref, lse_ref = ref.attn_fwd(f64(inp.q), f64(inp.k), f64(inp.v), bias=f64(inp.bias), causal=causal,
                                  scale=scale, dropout=dropout)
    atol, rtol = TOL[dtype]
    assert_close(out.float().cpu().numpy(), o_ref, atol, rtol, "O")
    assert_close(lse.cpu().numpy(), lse_ref, LSE_ATOL, 0.0, "lse")


def check_fwd_sampled(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=False, bias=False, rows=64, seed=0, scale=None,
                      dropout=None):
    """Large shapes: the oracle computes `rows` seeded query rows per head, one by one."""
    inp = make_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, bias=bias, seed=seed)
    scale = D ** -0.5 if scale is None else scale
    out, lse = gpu_fwd(inp, causal, scale, dropout=dropout)
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    q, k, v, bb = f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.bias)
    atol, rtol = TOL[dtype]
    for b in range(B):
        for h in range(Hq):
            r = ref.sample_rows(Nq, rows, 1000 + h)
            o_ref, lse_ref = ref.attn_fwd_rows(q, k, v, b, h, r, bias=bb, causal=causal, scale=scale,
                                               dropout=dropout)
            assert_close(out[b, h, r], o_ref, atol, rtol, f"O[b={b},h={h}]")
            assert_close(lse[b, h, r], lse_ref, LSE_ATOL, 0.0, f"lse[b={b},h={h}]")
    return out, lse


def gpu_fwd_bwd(inp, causal, scale, dropout=None):
    dev = torch.device("cuda")
    q, k, v, do = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.do.to(dev)
    bias = None if inp.bias is None else inp.bias.to(dev)
    out, lse = attention_fwd(q, k, v, bias=bias, causal=causal, scale=scale, **_drop_kw(dropout))
    dq, dk, dv = attention_bwd(q, k, v, out, lse, do, bias=bias, causal=causal, scale=scale, **_drop_kw(dropout))
    torch.cuda.synchronize()
    assert ffpa_check_status() == 0
    return out, lse, dq, dk, dv


def check_bwd_full(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=False, bias=False, seed=0, dropout=None):
    inp = make_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, bias=bias, grad=True, seed=seed)
    scale = D ** -0.5
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale, dropout=dropout)
    gq, gk, gv = ref.attn_bwd(f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.do), bias=f64(inp.bias),
                              causal=causal, scale=scale, dropout=dropout)
    errs, tiles = {}, {}
    for name, gpu, want in (("dQ", dq, gq), ("dK", dk, gk), ("dV", dv, gv)):
        g = gpu.float().cpu().numpy()
        errs[name] = rel_fro(g, want)
        tiles.update(tile_errors(g, want, name))
    worst = max(errs, key=errs.get)
    assert errs[worst] <= GRAD_RTOL, f"{worst} relative Frobenius error {errs[worst]:.3e} ({errs})"
    worst = max(tiles, key=tiles.get)
    assert tiles[worst] <= GRAD_RTOL, f"{worst} relative Frobenius error {tiles[worst]:.3e}"
    return errs


def check_bwd_sampled(B, Hq, Hkv, Nq, Nkv, D, dtype, causal=False, bias=False, rows=64, seed=0, dropout=None):
    inp = make_inputs(B, Hq, Hkv, Nq, Nkv, D, dtype, bias=bias, grad=True, seed=seed)
    scale = D ** -0.5
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale, dropout=dropout)
    dq, dk, dv = (x.float().cpu().numpy() for x in (dq, dk, dv))
    q, k, v, do, bb = f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.do), f64(inp.bias)
    errs = {}
    for b in range(B):
        for g in range(Hkv):
            kr = ref.sample_rows(Nkv, rows, 2000 + g)
            group = Hq // Hkv
            qrows = {h: ref.sample_rows(Nq, rows, 1000 + h) for h in range(g * group, (g + 1) * group)}
            sdq, sdk, sdv = ref.attn_bwd_sampled(q, k, v, do, b, g, qrows, kr, bias=bb, causal=causal, scale=scale,
                                                 dropout=dropout)
            for h in qrows:
                errs[f"dQ[{b},{h}]"] = rel_fro(dq[b, h, qrows[h]], sdq[h])
            errs[f"dK[{b},{g}]"] = rel_fro(dk[b, g, kr], sdk)
            errs[f"dV[{b},{g}]"] = rel_fro(dv[b, g, kr], sdv)
    worst = max(errs, key=errs.get)
    assert errs[worst] <= GRAD_RTOL, f"{worst} relative Frobenius error {errs[worst]:.3e}"
    return errs
