"""Pins for the fp64 oracle, against facts that do not come from the oracle itself.

Each pin is a closed form, an invariant of the mathematics, an independent
library routine (PyTorch's scaled_dot_product_attention and autograd, in fp64
on the CPU) or brute force (central finite differences).  The last test plants
plausible mistakes in copies of the oracle and checks that some pin fails for
each, so the pins are known to bite.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle.attn_ref as ref

RNG = np.random.default_rng(1234)


def rand(*shape):
    return RNG.standard_normal(shape)


# ---------------------------------------------------------------- pins as functions
def pin_rows_sum_to_one(m=ref):
    q, k = rand(1, 2, 9, 8), rand(1, 1, 11, 8)
    for causal in (False, True):
        s = m.scores_head(q, k, rand(1, 1, 1, 11), 0, 1, 0, 0.3, causal)
        p, _ = m.probs_head(s)
        assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(p >= 0)


def pin_constant_v(m=ref):
    q, k = rand(2, 2, 7, 16), rand(2, 2, 13, 16)
    v = np.full((2, 2, 13, 16), 0.0) + np.arange(16)[None, None, None, :] * 0.5 - 1.0
    for causal in (False, True):
        o, _ = m.attn_fwd(q, k, v, bias=rand(1, 1, 1, 13), causal=causal)
        assert np.allclose(o, v[:, :, :1, :].repeat(7, axis=2), atol=1e-12)


def pin_zero_q(m=ref):
    # Q = 0: every visible key gets weight exp(bias_j) / sum; without bias the mean.
    n, nkv, d = 6, 10, 8
    q, k, v = np.zeros((1, 1, n, d)), rand(1, 1, nkv, d), rand(1, 1, nkv, d)
    o, lse = m.attn_fwd(q, k, v, causal=False)
    assert np.allclose(o[0, 0], v[0, 0].mean(axis=0)[None, :], atol=1e-12)
    assert np.allclose(lse, math.log(nkv), atol=1e-12)
    o, lse = m.attn_fwd(q, k, v, causal=True)
    for i in range(n):
        assert np.allclose(o[0, 0, i], v[0, 0, : i + 1].mean(axis=0), atol=1e-12)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-12
    bias = rand(1, 1, 1, nkv)
    o, lse = m.attn_fwd(q, k, v, bias=bias)
    w = np.exp(bias[0, 0, 0])
    assert np.allclose(o[0, 0], (w @ v[0, 0] / w.sum())[None, :], atol=1e-12)
    assert np.allclose(lse, math.log(nkv) + math.log(np.mean(w)), atol=1e-12)


def pin_causal_row0(m=ref):
    q, k, v = rand(1, 1, 5, 8), rand(1, 1, 5, 8), rand(1, 1, 5, 8)
    bias = rand(1, 1, 1, 5)
    scale = 0.37
    o, lse = m.attn_fwd(q, k, v, bias=bias, causal=True, scale=scale)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-12)
    assert abs(lse[0, 0, 0] - (scale * q[0, 0, 0] @ k[0, 0, 0] + bias[0, 0, 0, 0])) < 1e-12


def pin_single_key(m=ref):
    q, k, v = rand(1, 2, 4, 8), rand(1, 2, 1, 8), rand(1, 2, 1, 8)
    o, lse = m.attn_fwd(q, k, v)
    assert np.allclose(o, np.broadcast_to(v, o.shape), atol=1e-12)
    assert np.allclose(lse[0, 1], q[0, 1] @ k[0, 1, 0] / math.sqrt(8), atol=1e-12)


def pin_bias_shift(m=ref):
    q, k, v = rand(1, 1, 6, 8), rand(1, 1, 9, 8), rand(1, 1, 9, 8)
    bias = rand(1, 1, 1, 9)
    o1, l1 = m.attn_fwd(q, k, v, bias=bias)
    o2, l2 = m.attn_fwd(q, k, v, bias=bias + 2.5)
    assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1 + 2.5, l2, atol=1e-12)


def pin_permutation(m=ref):
    q, k, v = rand(1, 1, 6, 8), rand(1, 1, 9, 8), rand(1, 1, 9, 8)
    perm = RNG.permutation(9)
    o1, l1 = m.attn_fwd(q, k, v)
    o2, l2 = m.attn_fwd(q, k[:, :, perm], v[:, :, perm])
    assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)


def pin_gqa_repeat_interleave(m=ref):
    q, k, v = rand(2, 6, 7, 8), rand(2, 2, 9, 8), rand(2, 2, 9, 8)
    do = rand(2, 6, 7, 8)
    ke = torch.from_numpy(k).repeat_interleave(3, dim=1).numpy()
    ve = torch.from_numpy(v).repeat_interleave(3, dim=1).numpy()
    for causal in (False, True):
        o1, l1 = m.attn_fwd(q, k, v, causal=causal)
        o2, l2 = m.attn_fwd(q, ke, ve, causal=causal)
        assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)
        g1 = m.attn_bwd(q, k, v, do, causal=causal)
        g2 = m.attn_bwd(q, ke, ve, do, causal=causal)
        assert np.allclose(g1[0], g2[0], atol=1e-12)
        # the group's gradient is the sum over its expanded heads
        assert np.allclose(g1[1], g2[1].reshape(2, 2, 3, 9, 8).sum(axis=2), atol=1e-12)
        assert np.allclose(g1[2], g2[2].reshape(2, 2, 3, 9, 8).sum(axis=2), atol=1e-12)


def _torch_sdpa(q, k, v, bias, causal, scale, gqa):
    t = lambda x: torch.from_numpy(np.array(x, dtype=np.float64, copy=True))
    mask = None if bias is None else t(np.broadcast_to(bias, (q.shape[0], q.shape[1], q.shape[2], k.shape[2])))
    if causal:
        tri = torch.ones(q.shape[2], k.shape[2], dtype=torch.bool).tril()
        cm = torch.zeros(q.shape[2], k.shape[2], dtype=torch.float64).masked_fill(~tri, float("-inf"))
        mask = cm if mask is None else mask + cm
    return torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), attn_mask=mask, scale=scale, enable_gqa=gqa)


def pin_torch_sdpa(m=ref):
    # torch's is_causal is top-left; the explicit lower-triangular mask says the same.
    for (b, hq, hkv, nq, nkv, d, causal, use_bias) in [
        (1, 1, 1, 5, 5, 4, False, False), (2, 4, 2, 7, 11, 8, False, True),
        (1, 2, 2, 9, 9, 16, True, False), (1, 4, 1, 6, 10, 8, True, True),
        (1, 1, 1, 1, 13, 8, False, True),
    ]:
        q, k, v = rand(b, hq, nq, d), rand(b, hkv, nkv, d), rand(b, hkv, nkv, d)
        bias = rand(1, 1, 1, nkv) if use_bias else None
        scale = 1.0 / math.sqrt(d)
        o, lse = m.attn_fwd(q, k, v, bias=bias, causal=causal)
        ot = _torch_sdpa(q, k, v, bias, causal, scale, hq != hkv).numpy()
        assert np.allclose(o, ot, atol=1e-12, rtol=1e-12)
        # lse against torch.logsumexp of independently formed scores
        kt = torch.from_numpy(k).repeat_interleave(hq // hkv, dim=1)
        st = torch.from_numpy(q) @ kt.transpose(-1, -2) * scale
        if bias is not None:
            st = st + torch.from_numpy(bias)
        if causal:
            st = st.masked_fill(~torch.ones(nq, nkv, dtype=torch.bool).tril(), float("-inf"))
        assert np.allclose(lse, torch.logsumexp(st, dim=-1).numpy(), atol=1e-12)


def pin_torch_autograd(m=ref):
    for (hq, hkv, nq, nkv, d, causal, use_bias) in [
        (2, 1, 5, 7, 4, False, True), (2, 2, 6, 6, 8, True, False), (4, 2, 3, 9, 8, True, True)]:
        q, k, v, do = rand(1, hq, nq, d), rand(1, hkv, nkv, d), rand(1, hkv, nkv, d), rand(1, hq, nq, d)
        bias = rand(1, 1, 1, nkv) if use_bias else None
        tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
        mask = None if bias is None else torch.from_numpy(bias)
        if causal:
            cm = torch.zeros(nq, nkv, dtype=torch.float64).masked_fill(
                ~torch.ones(nq, nkv, dtype=torch.bool).tril(), float("-inf"))
            mask = cm if mask is None else mask + cm
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, enable_gqa=hq != hkv)
        out.backward(torch.from_numpy(do))
        dq, dk, dv = m.attn_bwd(q, k, v, do, bias=bias, causal=causal)
        assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
        assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
        assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)


def pin_finite_differences(m=ref):
    # B=1, Hq=2, Hkv=1, N=5, D=4: central differences of L = sum(O * dO)
    q, k, v, do = rand(1, 2, 5, 4), rand(1, 1, 5, 4), rand(1, 1, 5, 4), rand(1, 2, 5, 4)
    bias = rand(1, 1, 1, 5)
    for causal in (False, True):
        loss = lambda q_, k_, v_: float(np.sum(m.attn_fwd(q_, k_, v_, bias=bias, causal=causal)[0] * do))
        grads = m.attn_bwd(q, k, v, do, bias=bias, causal=causal)
        h = 1e-6
        for which, x in enumerate((q, k, v)):
            num = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][idx] += h
                args_m[which][idx] -= h
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            err = np.linalg.norm(grads[which] - num) / np.linalg.norm(num)
            assert err < 1e-6, (which, causal, err)


def pin_bwd_sums(m=ref):
    q, k, v, do = rand(2, 4, 7, 8), rand(2, 2, 9, 8), rand(2, 2, 9, 8), rand(2, 4, 7, 8)
    for causal in (False, True):
        dq, dk, dv = m.attn_bwd(q, k, v, do, bias=rand(1, 1, 1, 9), causal=causal)
        assert np.allclose(dk.sum(axis=2), 0.0, atol=1e-12)
        assert np.allclose(dv.sum(axis=2), do.reshape(2, 2, 2, 7, 8).sum(axis=(2, 3)), atol=1e-12)


def pin_sampled_bwd(m=ref):
    q, k, v, do = rand(1, 4, 37, 8), rand(1, 2, 41, 8), rand(1, 2, 41, 8), rand(1, 4, 37, 8)
    bias = rand(1, 1, 1, 41)
    for causal in (False, True):
        dq, dk, dv = m.attn_bwd(q, k, v, do, bias=bias, causal=causal)
        qr, kr = m.sample_rows(37, 6, 3), m.sample_rows(41, 5, 4)
        for g in range(2):
            sdq, sdk, sdv = m.attn_bwd_sampled(q, k, v, do, 0, g, qr, kr, bias=bias, causal=causal, block=8)
            for h, val in sdq.items():
                assert np.allclose(val, dq[0, h, qr], atol=1e-12)
            assert np.allclose(sdk, dk[0, g, kr], atol=1e-12)
            assert np.allclose(sdv, dv[0, g, kr], atol=1e-12)
        o, lse = m.attn_fwd(q, k, v, bias=bias, causal=causal)
        orow, lrow = m.attn_fwd_rows(q, k, v, 0, 3, qr, bias=bias, causal=causal)
        assert np.allclose(orow, o[0, 3, qr], atol=1e-12) and np.allclose(lrow, lse[0, 3, qr], atol=1e-12)


def pin_query_bias(m=ref):
    # a [1,1,Nq,Nkv] bias whose rows are equal is the [1,1,1,Nkv] bias
    q, k, v = rand(1, 2, 5, 8), rand(1, 2, 7, 8), rand(1, 2, 7, 8)
    row = rand(1, 1, 1, 7)
    o1, l1 = m.attn_fwd(q, k, v, bias=row)
    o2, l2 = m.attn_fwd(q, k, v, bias=np.repeat(row, 5, axis=2))
    assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)


def pin_torch_bias_broadcast(m=ref):
    # Every broadcast form of the additive bias ([1,1,Nq,Nkv] per-query, [B,Hq,1,Nkv],
    # [B,1,Nq,Nkv], [1,Hq,Nq,Nkv], [B,Hq,Nq,Nkv]) with distinct rows, heads and batches,
    # against torch SDPA and autograd in fp64 (torch broadcasts the float mask itself);
    # then the row-sampled forms of the oracle on the same biases against its full forms.
    b, hq, hkv, nq, nkv, d = 2, 4, 2, 6, 9, 8
    q, k, v, do = rand(b, hq, nq, d), rand(b, hkv, nkv, d), rand(b, hkv, nkv, d), rand(b, hq, nq, d)
    scale = 1.0 / math.sqrt(d)
    for shape in [(1, 1, nq, nkv), (b, hq, 1, nkv), (b, 1, nq, nkv), (1, hq, nq, nkv), (b, hq, nq, nkv)]:
        bias = rand(*shape)
        for causal in (False, True):
            o, lse = m.attn_fwd(q, k, v, bias=bias, causal=causal)
            tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
            mask = torch.from_numpy(bias.copy())
            if causal:
                mask = mask + torch.zeros(nq, nkv, dtype=torch.float64).masked_fill(
                    ~torch.ones(nq, nkv, dtype=torch.bool).tril(), float("-inf"))
            out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale,
                                                                   enable_gqa=True)
            assert np.allclose(o, out.detach().numpy(), atol=1e-12, rtol=1e-12), (shape, causal)
            st = (torch.from_numpy(q) @ torch.from_numpy(k).repeat_interleave(hq // hkv, dim=1).transpose(-1, -2)
                  * scale + mask)
            assert np.allclose(lse, torch.logsumexp(st, dim=-1).numpy(), atol=1e-12), (shape, causal)
            out.backward(torch.from_numpy(do))
            dq, dk, dv = m.attn_bwd(q, k, v, do, bias=bias, causal=causal)
            for mine, theirs in ((dq, tq), (dk, tk), (dv, tv)):
                assert np.allclose(mine, theirs.grad.numpy(), atol=1e-11), (shape, causal)
            rows = np.array([4, 1, 5])
            for bi in range(b):
                for h in range(hq):
                    orow, lrow = m.attn_fwd_rows(q, k, v, bi, h, rows, bias=bias, causal=causal)
                    assert np.allclose(orow, o[bi, h, rows], atol=1e-12), (shape, causal, bi, h)
                    assert np.allclose(lrow, lse[bi, h, rows], atol=1e-12), (shape, causal, bi, h)
            kr = np.array([8, 0, 3])
            for bi in range(b):
                for g in range(hkv):
                    sdq, sdk, sdv = m.attn_bwd_sampled(q, k, v, do, bi, g, rows, kr, bias=bias, causal=causal,
                                                       block=4)
                    for h, val in sdq.items():
                        assert np.allclose(val, dq[bi, h, rows], atol=1e-12), (shape, causal, bi, h)
                    assert np.allclose(sdk, dk[bi, g, kr], atol=1e-12), (shape, causal, bi, g)
                    assert np.allclose(sdv, dv[bi, g, kr], atol=1e-12), (shape, causal, bi, g)


def pin_philox_known_answers(m=ref):
    # the generator against the published known-answer vectors
    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        out = m.philox4x32_10(w[0:4], w[4:6])
        assert [int(x) for x in out] == w[6:10], r


def pin_dropout_layout(m=ref):
    # the keep mask's layout, element by element: score (i, j) of query head h in
    # batch b reads 16-bit field j % 2 of word (j % 8) // 2 of the generator's
    # output at counter (j // 8, i, b * Hq + h, offset), key = (seed lo, seed hi)
    p, seed, offset, hq = 0.37, 0x0123456789ABCDEF, 5, 3
    t = m.dropout_threshold(p)
    assert t == 24248                                    # floor(0.37 * 65536 + 1/2)
    rows, cols = np.array([0, 1, 7, 130, 8191]), np.array([0, 1, 2, 7, 8, 9, 63, 100, 8190])
    for b, h in ((0, 0), (1, 2)):
        keep = m.dropout_keep(b, h, hq, rows, cols, p, seed, offset)
        for a, i in enumerate(rows):
            for c, j in enumerate(cols):
                x = m.philox4x32_10((int(j) // 8, int(i), b * hq + h, offset),
                                    (seed & 0xFFFFFFFF, seed >> 32))
                u = (int(x[(int(j) % 8) // 2]) >> (16 * (int(j) % 2))) & 0xFFFF
                assert bool(keep[a, c]) == (u >= t), (b, h, i, j)


def pin_dropout_rate(m=ref):
    # the kept fraction is 1 - t / 65536 within 6 sigma; p = 0 keeps every score;
    # other heads, batches and offsets draw other masks
    n_r, n_c = 128, 2048
    for p in (0.1, 0.5, 0.9):
        keep = m.dropout_keep(0, 1, 4, np.arange(n_r), np.arange(n_c), p, 99, 0)
        q = 1.0 - m.dropout_threshold(p) / 65536.0
        sigma = math.sqrt(q * (1 - q) / keep.size)
        assert abs(keep.mean() - q) < 6 * sigma, (p, keep.mean(), q)
        for other in (m.dropout_keep(0, 2, 4, np.arange(n_r), np.arange(n_c), p, 99, 0),
                      m.dropout_keep(1, 1, 4, np.arange(n_r), np.arange(n_c), p, 99, 0),
                      m.dropout_keep(0, 1, 4, np.arange(n_r), np.arange(n_c), p, 99, 1),
                      m.dropout_keep(0, 1, 4, np.arange(n_r), np.arange(n_c), p, 98, 0)):
            # two independent masks differ at a fraction 2 q (1 - q) of the scores
            diff = float(np.mean(keep != other))
            assert abs(diff - 2 * q * (1 - q)) < 0.02, (p, diff)
    assert m.dropout_keep(0, 0, 1, np.arange(64), np.arange(64), 0.0, 5, 0).all()


def _torch_dropout_attention(q, k, v, bias, causal, scale, z):
    # fp64 autograd through softmax, a fixed multiplier Z on P, and P V
    tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
    hq, hkv, nq, nkv = q.shape[1], k.shape[1], q.shape[2], k.shape[2]
    kk = tk.repeat_interleave(hq // hkv, dim=1)
    vv = tv.repeat_interleave(hq // hkv, dim=1)
    s = tq @ kk.transpose(-1, -2) * scale
    if bias is not None:
        s = s + torch.from_numpy(bias)
    if causal:
        s = s.masked_fill(~torch.ones(nq, nkv, dtype=torch.bool).tril(), float("-inf"))
    pz = torch.softmax(s, dim=-1) * torch.from_numpy(z)
    return tq, tk, tv, pz @ vv, torch.logsumexp(s, dim=-1)


def pin_dropout_torch_autograd(m=ref):
    # forward and gradients with dropout against PyTorch autograd in fp64, the
    # multiplier Z = keep / (1 - p) taken from the layout-pinned keep mask; the
    # row-sampled forms against the full ones
    for (bsz, hq, hkv, nq, nkv, d, causal, use_bias) in [
            (1, 2, 1, 7, 19, 8, False, True), (2, 2, 2, 9, 9, 4, True, False), (1, 4, 2, 6, 17, 8, True, True)]:
        q, k, v, do = rand(bsz, hq, nq, d), rand(bsz, hkv, nkv, d), rand(bsz, hkv, nkv, d), rand(bsz, hq, nq, d)
        bias = rand(1, 1, 1, nkv) if use_bias else None
        drop = (0.3, 0xDEADBEEF12345678, 3)
        z = np.zeros((bsz, hq, nq, nkv))
        for b in range(bsz):
            for h in range(hq):
                z[b, h] = m.dropout_keep(b, h, hq, np.arange(nq), np.arange(nkv), *drop) / 0.7
        assert 0 < np.count_nonzero(z) < z.size
        scale = 1.0 / math.sqrt(d)
        tq, tk, tv, out, lse_t = _torch_dropout_attention(q, k, v, bias, causal, scale, z)
        o, lse = m.attn_fwd(q, k, v, bias=bias, causal=causal, dropout=drop)
        assert np.allclose(o, out.detach().numpy(), atol=1e-12), (nq, nkv, causal)
        assert np.allclose(lse, lse_t.detach().numpy(), atol=1e-12)
        out.backward(torch.from_numpy(do))
        dq, dk, dv = m.attn_bwd(q, k, v, do, bias=bias, causal=causal, dropout=drop)
        for mine, theirs in ((dq, tq), (dk, tk), (dv, tv)):
            assert np.allclose(mine, theirs.grad.numpy(), atol=1e-11), (nq, nkv, causal)
        rows, kr = np.array([nq - 1, 0, 2]), np.array([nkv - 1, 1, 4])
        orow, lrow = m.attn_fwd_rows(q, k, v, bsz - 1, hq - 1, rows, bias=bias, causal=causal, dropout=drop)
        assert np.allclose(orow, o[bsz - 1, hq - 1, rows], atol=1e-12)
        for g in range(hkv):
            sdq, sdk, sdv = m.attn_bwd_sampled(q, k, v, do, bsz - 1, g, rows, kr, bias=bias, causal=causal,
                                               block=4, dropout=drop)
            for h, val in sdq.items():
                assert np.allclose(val, dq[bsz - 1, h, rows], atol=1e-12)
            assert np.allclose(sdk, dk[bsz - 1, g, kr], atol=1e-12)
            assert np.allclose(sdv, dv[bsz - 1, g, kr], atol=1e-12)
        # p = 0 is the plain attention
        o0, _ = m.attn_fwd(q, k, v, bias=bias, causal=causal, dropout=(0.0, 1, 0))
        assert np.allclose(o0, m.attn_fwd(q, k, v, bias=bias, causal=causal)[0], atol=1e-14)


PINS = [pin_rows_sum_to_one, pin_constant_v, pin_zero_q, pin_causal_row0, pin_single_key, pin_bias_shift,
        pin_permutation, pin_gqa_repeat_interleave, pin_torch_sdpa, pin_torch_autograd, pin_finite_differences,
        pin_bwd_sums, pin_sampled_bwd, pin_query_bias, pin_torch_bias_broadcast, pin_philox_known_answers,
        pin_dropout_layout, pin_dropout_rate, pin_dropout_torch_autograd]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_dead_row_convention():
    # reading: a row with every score at -inf gives P = 0 and lse = -inf
    s = np.array([[-np.inf, -np.inf], [0.0, 1.0]])
    p, lse = ref.probs_head(s)
    assert np.all(p[0] == 0) and lse[0] == -np.inf
    assert np.allclose(p[1].sum(), 1.0)


def test_sample_rows():
    r = ref.sample_rows(8192, 64, 1000)
    assert len(r) == 64 and len(set(r.tolist())) == 64 and r[0] == 0 and r[-1] == 8191
    assert np.array_equal(r, ref.sample_rows(8192, 64, 1000))
    assert np.array_equal(ref.sample_rows(10, 64, 0), np.arange(10))


def test_lse_magnitude():
    # N(0,1) inputs with scale 1/sqrt(D): scores ~ N(0,1), lse ~ ln N + 1/2 (loose sanity range)
    q, k, v = rand(1, 1, 64, 512), rand(1, 1, 256, 512), rand(1, 1, 256, 512)
    _, lse = ref.attn_fwd(q, k, v)
    assert abs(lse.mean() - (math.log(256) + 0.5)) < 0.3


# ---------------------------------------------------------------- the pins bite
def _mutant_module(**over):
    import importlib.util
    # a fresh copy of the oracle module inside the oracle package (its relative imports resolve)
    spec = importlib.util.spec_from_file_location("oracle.attn_ref_mutant", ref.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    for name, fn in over.items():
        setattr(mod, name, fn(mod))
    return mod


def _mut_no_scale(mod):
    orig = mod.scores_head
    return lambda q, k, bias, b, h, g, scale, causal, rows=None, cols=None: orig(q, k, bias, b, h, g, 1.0, causal, rows, cols)


def _mut_causal_flipped(mod):
    orig = mod.scores_head

    def f(q, k, bias, b, h, g, scale, causal, rows=None, cols=None):
        if not causal:
            return orig(q, k, bias, b, h, g, scale, False, rows, cols)
        s = orig(q, k, bias, b, h, g, scale, False, rows, cols)
        r = np.arange(q.shape[2]) if rows is None else np.asarray(rows)
        c = np.arange(k.shape[2]) if cols is None else np.asarray(cols)
        return np.where(c[None, :] < r[:, None], -np.inf, s)
    return f


def _mut_gqa_modulo(mod):
    return lambda h, hq, hkv: h % hkv


def _mut_lse_log2(mod):
    orig = mod.probs_head

    def f(s):
        p, lse = orig(s)
        return p, lse / math.log(2)
    return f


def _mut_bias_sign(mod):
    orig = mod._bias_rows
    return lambda bias, b, h, rows, nkv: (lambda r: r if np.isscalar(r) else -r)(orig(bias, b, h, rows, nkv))


def _mut_bwd_delta_dropped(mod):
    def f(q, k, v, do, bias=None, causal=False, scale=None):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        scale = 1.0 / math.sqrt(q.shape[3]) if scale is None else scale
        dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                g = mod.kv_head_of(h, q.shape[1], k.shape[1])
                p, _ = mod.probs_head(mod.scores_head(q, k, bias, b, h, g, scale, causal))
                dv[b, g] += p.T @ do[b, h]
                ds = p * (do[b, h] @ v[b, g].T)          # Delta term dropped
                dq[b, h] = scale * (ds @ k[b, g])
                dk[b, g] += scale * (ds.T @ q[b, h])
        return dq, dk, dv
    return f


def _mut_pv_transposed_v(mod):
    orig = mod.attn_fwd

    def f(q, k, v, bias=None, causal=False, scale=None):
        v = np.asarray(v, dtype=np.float64)
        if v.shape[2] == v.shape[3]:
            v = np.swapaxes(v, 2, 3)
        else:
            v = v[:, :, ::-1]                             # wrong row order instead
        return orig(q, k, v, bias, causal, scale)
    return f


def _mut_sampled_dk_unscaled(mod):
    orig = mod.attn_bwd_sampled

    def f(q, k, v, do, b, h_kv, q_rows, kv_rows, bias=None, causal=False, scale=None, block=1024):
        dq, dk, dv = orig(q, k, v, do, b, h_kv, q_rows, kv_rows, bias, causal, scale, block)
        s = 1.0 / math.sqrt(np.shape(q)[3]) if scale is None else scale
        return dq, dk / s, dv                             # scale dropped from dK
    return f


def _mut_sampled_dv_one_head(mod):
    orig = mod.attn_bwd_sampled

    def f(q, k, v, do, b, h_kv, q_rows, kv_rows, bias=None, causal=False, scale=None, block=1024):
        # dV from the group's first query head only, scaled up: GQA sum replaced by a copy
        q, do = np.asarray(q, dtype=np.float64), np.asarray(do, dtype=np.float64)
        group = q.shape[1] // np.shape(k)[1]
        first = h_kv * group
        qq, dd = q.copy(), do.copy()
        for h in range(first + 1, first + group):
            qq[:, h], dd[:, h] = q[:, first], do[:, first]
        dq, dk, _ = orig(q, k, v, do, b, h_kv, q_rows, kv_rows, bias, causal, scale, block)
        _, _, dv = orig(qq, k, v, dd, b, h_kv, q_rows, kv_rows, bias, causal, scale, block)
        return dq, dk, dv
    return f


def _mut_fwd_rows_next_head(mod):
    orig = mod.attn_fwd_rows

    def f(q, k, v, b, h, rows, bias=None, causal=False, scale=None):
        return orig(q, k, v, b, (h + 1) % np.shape(q)[1], rows, bias, causal, scale)
    return f


def _bias_head(mod, pick_rows):
    # _bias_rows with the broadcast done by hand, so a mutant can change one index
    def f(bias, b, h, rows, nkv):
        if bias is None:
            return 0.0
        bias = np.asarray(bias, dtype=np.float64)
        bb = bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0]
        return pick_rows(bb, np.asarray(rows), nkv)
    return f


def _mut_bias_first_row(mod):
    # a per-query bias read as if its first row applied to every query
    return _bias_head(mod, lambda bb, rows, nkv: np.broadcast_to(bb[0], (len(rows), nkv)))


def _mut_bias_row_shifted(mod):
    # a per-query bias read one row late (clamped at the last row)
    return _bias_head(mod, lambda bb, rows, nkv: bb[np.minimum(rows + 1, bb.shape[0] - 1)]
                      if bb.shape[0] > 1 else np.broadcast_to(bb[0], (len(rows), nkv)))


def _mut_bias_head_ignored(mod):
    orig = mod._bias_rows
    return lambda bias, b, h, rows, nkv: orig(bias, b, 0, rows, nkv)


def _mut_bias_batch_ignored(mod):
    orig = mod._bias_rows
    return lambda bias, b, h, rows, nkv: orig(bias, 0, h, rows, nkv)


def _mut_philox_nine_rounds(mod):
    def f(counter, key):
        c = [np.asarray(x, dtype=np.uint64) & np.uint64(0xFFFFFFFF) for x in counter]
        c = list(np.broadcast_arrays(*c))
        k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
        for r in range(9):                                # one round short
            if r:
                k0, k1 = (k0 + 0x9E3779B9) & 0xFFFFFFFF, (k1 + 0xBB67AE85) & 0xFFFFFFFF
            p0, p1 = np.uint64(0xD2511F53) * c[0], np.uint64(0xCD9E8D57) * c[2]
            c = [(p1 >> np.uint64(32)) ^ c[1] ^ np.uint64(k0), p1 & np.uint64(0xFFFFFFFF),
                 (p0 >> np.uint64(32)) ^ c[3] ^ np.uint64(k1), p0 & np.uint64(0xFFFFFFFF)]
        return c
    return f


def _mut_dropout_field(mod):
    # the 16-bit field picked as word j % 4, half (j // 4) % 2
    def f(b, h, hq, rows, cols, p, seed, offset):
        t = mod.dropout_threshold(p)
        i = np.asarray(rows, dtype=np.uint64)[:, None]
        j = np.asarray(cols, dtype=np.uint64)[None, :]
        x = mod.philox4x32_10((j >> np.uint64(3), i, b * hq + h, offset), (seed & 0xFFFFFFFF, seed >> 32))
        jm = (j & np.uint64(7)) + np.zeros_like(i)
        word = np.choose((jm & np.uint64(3)).astype(np.int64), x)
        return ((word >> (np.uint64(16) * (jm >> np.uint64(2)))) & np.uint64(0xFFFF)) >= np.uint64(t)
    return f


def _mut_dropout_head_ignored(mod):
    orig = mod.dropout_keep
    return lambda b, h, hq, rows, cols, p, seed, offset: orig(b, 0, hq, rows, cols, p, seed, offset)


def _mut_dropout_dp_unmasked(mod):
    orig = mod.attn_bwd

    def f(q, k, v, do, bias=None, causal=False, scale=None, dropout=None):
        if dropout is None:
            return orig(q, k, v, do, bias, causal, scale)
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        scale = 1.0 / math.sqrt(q.shape[3]) if scale is None else scale
        hq = q.shape[1]
        dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        for b in range(q.shape[0]):
            for h in range(hq):
                g = mod.kv_head_of(h, hq, k.shape[1])
                p, _ = mod.probs_head(mod.scores_head(q, k, bias, b, h, g, scale, causal))
                z = mod.dropout_keep(b, h, hq, np.arange(q.shape[2]), np.arange(k.shape[2]), *dropout) / (
                    1.0 - dropout[0])
                o = (p * z) @ v[b, g]
                dv[b, g] += (p * z).T @ do[b, h]
                dp = do[b, h] @ v[b, g].T                 # Z left out of dP
                ds = p * (dp - np.sum(do[b, h] * o, axis=1)[:, None])
                dq[b, h] = scale * (ds @ k[b, g])
                dk[b, g] += scale * (ds.T @ q[b, h])
        return dq, dk, dv
    return f


MUTANTS = {
    "no_scale": {"scores_head": _mut_no_scale},
    "causal_flipped": {"scores_head": _mut_causal_flipped},
    "gqa_modulo": {"kv_head_of": _mut_gqa_modulo},
    "lse_log2": {"probs_head": _mut_lse_log2},
    "bias_sign": {"_bias_rows": _mut_bias_sign},
    "bwd_delta_dropped": {"attn_bwd": _mut_bwd_delta_dropped},
    "pv_wrong_v": {"attn_fwd": _mut_pv_transposed_v},
    "sampled_dk_unscaled": {"attn_bwd_sampled": _mut_sampled_dk_unscaled},
    "sampled_dv_one_head": {"attn_bwd_sampled": _mut_sampled_dv_one_head},
    "fwd_rows_next_head": {"attn_fwd_rows": _mut_fwd_rows_next_head},
    "bias_first_row": {"_bias_rows": _mut_bias_first_row},
    "bias_row_shifted": {"_bias_rows": _mut_bias_row_shifted},
    "bias_head_ignored": {"_bias_rows": _mut_bias_head_ignored},
    "bias_batch_ignored": {"_bias_rows": _mut_bias_batch_ignored},
    "philox_nine_rounds": {"philox4x32_10": _mut_philox_nine_rounds},
    "dropout_field": {"dropout_keep": _mut_dropout_field},
    "dropout_head_ignored": {"dropout_keep": _mut_dropout_head_ignored},
    "dropout_dp_unmasked": {"attn_bwd": _mut_dropout_dp_unmasked},
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    mod = _mutant_module(**MUTANTS[name])
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except AssertionError:
            caught.append(pin.__name__)
        except Exception:
            caught.append(pin.__name__ + "!")
    assert caught, f"no pin catches mutant {name}"


@pytest.mark.parametrize("name", ["bias_first_row", "bias_row_shifted", "bias_head_ignored", "bias_batch_ignored"])
def test_bias_broadcast_mutants_need_the_broadcast_pin(name):
    # These mistakes in the per-query / per-head / per-batch bias branches slip past
    # every pin that uses a key-position bias or equal rows; the broadcast pin alone
    # catches them.
    mod = _mutant_module(**MUTANTS[name])
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught == ["pin_torch_bias_broadcast"], caught
