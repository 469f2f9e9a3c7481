"""Pins that tie the fp64 oracle to facts outside itself.

Page shorthand: [P1] "【多模态大模型】FlashAttention in NeurIPS 2022" (coreui.cn);
[P2] "FlashAttention" notes (maosong.website); [P3] "Transformer 入门"
(cansult.github.io); [P4] "Как работает FlashAttention математически" (aivaro.ru).

Each pin takes the oracle module and raises AssertionError when the oracle
disagrees with: the pages' worked example, a closed form, an invariant the
pages prove, central finite differences, or PyTorch's own fp64 attention
routine with an independently built mask.  The mutation tests run the same
pins against deliberately broken copies of the oracle and require a failure,
so a plausible slip (dropped term, wrong sign or index, transposed operand)
cannot pass unnoticed.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _dense_mask_torch(N, causal=False, block_mask=None, block=128):
    """Boolean [N, N] visibility built with torch ops, independently of the oracle."""
    m = torch.ones(N, N, dtype=torch.bool)
    if causal:
        m = torch.tril(m)
    if block_mask is not None:
        bm = torch.as_tensor(np.asarray(block_mask)).bool()
        m = m & bm.repeat_interleave(block, 0).repeat_interleave(block, 1)[:N, :N]
    return m


# --------------------------------------------------------------------------- #
def pin_worked_example(orc):
    """[P1 2.1] softmax([1,2,3,10]) in two blocks; V=[[1,2],[3,4],[5,6],[7,8]]."""
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    s = np.array(g["scores"])
    V = np.array(g["V"])
    # q . k_j = s_j with d = 1 and scale = 1 (the page applies no scale)
    q = np.ones((1, 1, 1, 1))
    k = s.reshape(1, 1, -1, 1)
    v = V.reshape(1, 1, *V.shape)
    o, lse = orc.forward(q, k, v, 1.0)
    to, tlse, traces = orc.tiled_forward(q, k, v, 1.0, Br=1, Bc=g["block"], trace=True)

    ex = [math.exp(e) for e in g["softmax_exponents"]]
    p_expect = np.array(ex) / sum(ex)
    p, lse_p = orc.head_probs(q[0, 0], k[0, 0], 1.0)
    np.testing.assert_allclose(p[0], p_expect, rtol=1e-14, atol=0)
    for step, st in zip(traces[0], g["after_block"]):
        m_t, l_t, o_t = step
        l_exp = sum(math.exp(e) for e in st["l_exponents"])
        o_exp = sum(math.exp(e) * V[r] for r, e in zip(st["o_rows"], st["o_exponents"])) / l_exp
        assert m_t[0] == st["m"]
        np.testing.assert_allclose(l_t[0], l_exp, rtol=1e-14)
        np.testing.assert_allclose(o_t[0], o_exp, rtol=1e-14)
    final = g["after_block"][-1]
    l_fin = sum(math.exp(e) for e in final["l_exponents"])
    o_fin = sum(math.exp(e) * V[r] for r, e in zip(final["o_rows"], final["o_exponents"])) / l_fin
    for oo in (o[0, 0, 0], to[0, 0, 0]):
        np.testing.assert_allclose(oo, o_fin, rtol=1e-14)
    for ll in (lse[0, 0, 0], tlse[0, 0, 0], lse_p[0]):
        np.testing.assert_allclose(ll, final["m"] + math.log(l_fin), rtol=1e-14)


# --------------------------------------------------------------------------- #
def pin_closed_forms(orc):
    r = _rng(1)
    B, H, N, d = 1, 2, 37, 8
    v = r.standard_normal((B, H, N, d))
    k = r.standard_normal((B, H, N, d))
    q0 = np.zeros((B, H, N, d))
    scale = 0.3
    # Q = 0: uniform weights -> O = mean of visible V rows, LSE = ln(#visible)
    o, lse = orc.forward(q0, k, v, scale)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-13)
    np.testing.assert_allclose(lse, np.full((B, H, N), math.log(N)), atol=1e-13)
    o, lse = orc.forward(q0, k, v, scale, causal=True)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix, atol=1e-13)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape), atol=1e-13)
    # block mask with block 4: row i sees the keys of its visible blocks
    bm = (r.random((10, 10)) < 0.4).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    o, lse = orc.forward(q0, k, v, scale, block_mask=bm, block=4)
    for i in range(N):
        keys = [j for j in range(N) if bm[i // 4, j // 4]]
        np.testing.assert_allclose(o[:, :, i], v[:, :, keys].mean(axis=2), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(len(keys)), atol=1e-13)
    # N = 1: O = V, LSE = scale * q . k
    q1 = r.standard_normal((1, 1, 1, 5))
    k1 = r.standard_normal((1, 1, 1, 5))
    v1 = r.standard_normal((1, 1, 1, 3))
    o, lse = orc.forward(q1, k1, v1, 0.7)
    np.testing.assert_allclose(o, v1, rtol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], 0.7 * float(q1.ravel() @ k1.ravel()), rtol=1e-14)
    # one key far above the rest: O equals that key's V row
    qp = np.full((1, 1, 6, 4), 1e3)
    kp = np.full((1, 1, 9, 4), -1.0)
    kp[0, 0, 5] = 1.0                      # q . k_5 = 4e3, every other q . k_j = -4e3
    vp = r.standard_normal((1, 1, 9, 3))
    o, _ = orc.forward(qp, kp, vp, 1.0)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(vp[0, 0, 5], (6, 3)), rtol=1e-12)


# --------------------------------------------------------------------------- #
def pin_invariants(orc):
    r = _rng(2)
    B, H, N, d = 2, 2, 45, 6
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    scale = 1 / math.sqrt(d)
    # rows of P sum to 1 [P1: softmax turns a row into a distribution]
    for causal in (False, True):
        p, lse = orc.head_probs(q[0, 1], k[0, 1], scale, causal=causal)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
        # LSE normalises exp(S): exp(S - LSE) reproduces P
        s = scale * q[0, 1] @ k[0, 1].T
        if causal:
            s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
        np.testing.assert_allclose(np.exp(s - lse[:, None]), p, atol=1e-14)
    # shift invariance: add c_i to row i of S through an extra feature column
    c = r.standard_normal(N) * 5
    qa = np.concatenate([q, np.broadcast_to(c[None, None, :, None], (B, H, N, 1))], axis=-1)
    ka = np.concatenate([k, np.full((B, H, N, 1), 1.0 / scale)], axis=-1)
    o0, l0 = orc.forward(q, k, v, scale)
    o1, l1 = orc.forward(qa, ka, v, scale)
    np.testing.assert_allclose(o1, o0, atol=1e-12)
    np.testing.assert_allclose(l1, l0 + c[None, None, :], atol=1e-12)
    # tiled == materialised for any split point (Theorem 1), incl. 1 and non-divisors
    bm = (r.random((12, 12)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    for causal, mask in ((False, None), (True, None), (False, bm)):
        ref_o, ref_l = orc.forward(q, k, v, scale, causal=causal, block_mask=mask, block=4)
        for Br, Bc in ((1, 1), (2, 3), (7, 16), (16, 7), (45, 45), (128, 128)):
            to, tl = orc.tiled_forward(q, k, v, scale, Br, Bc, causal=causal,
                                       block_mask=mask, block=4)
            np.testing.assert_allclose(to, ref_o, atol=1e-12)
            np.testing.assert_allclose(tl, ref_l, atol=1e-12)
    # merge of (m, l) is exact for every split point [P2 "Tiling"]
    x = r.standard_normal(40) * 4
    for cut in range(1, 40):
        a, b = x[:cut], x[cut:]
        m, l = orc.merge_stats(a.max(), np.exp(a - a.max()).sum(), b.max(), np.exp(b - b.max()).sum())
        assert m == x.max()
        np.testing.assert_allclose(l, np.exp(x - x.max()).sum(), rtol=1e-14)
    # causal row i == non-causal attention over keys 0..i
    oc, lc = orc.forward(q, k, v, scale, causal=True)
    for i in (0, 1, 17, N - 1):
        op, lp = orc.forward(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], scale)
        np.testing.assert_allclose(oc[:, :, i], op[:, :, 0], atol=1e-13)
        np.testing.assert_allclose(lc[:, :, i], lp[:, :, 0], atol=1e-13)
    # block mask of all ones == dense; diagonal-only == independent blocks
    Nb = 3 * 4
    qb, kb, vb = q[:, :, :Nb], k[:, :, :Nb], v[:, :, :Nb]
    od, ld = orc.forward(qb, kb, vb, scale)
    o1, l1 = orc.forward(qb, kb, vb, scale, block_mask=np.ones((3, 3), np.uint8), block=4)
    np.testing.assert_allclose(o1, od, atol=1e-14)
    np.testing.assert_allclose(l1, ld, atol=1e-14)
    o2, l2 = orc.forward(qb, kb, vb, scale, block_mask=np.eye(3, dtype=np.uint8), block=4)
    for blk in range(3):
        sl = slice(4 * blk, 4 * blk + 4)
        ob, lb = orc.forward(qb[:, :, sl], kb[:, :, sl], vb[:, :, sl], scale)
        np.testing.assert_allclose(o2[:, :, sl], ob, atol=1e-13)
        np.testing.assert_allclose(l2[:, :, sl], lb, atol=1e-13)
    # sampled-row helpers agree with the full computation
    rows = [0, 3, 44]
    orr, lrr = orc.forward_rows(q, k, v, scale, 1, 0, rows, causal=True)
    np.testing.assert_allclose(orr, oc[1, 0, rows], atol=1e-14)
    np.testing.assert_allclose(lrr, lc[1, 0, rows], atol=1e-14)


# --------------------------------------------------------------------------- #
def pin_backward_fd(orc):
    """Central finite differences of phi = sum(dO o O) on tiny inputs."""
    r = _rng(3)
    cases = [(3, 2, False, None), (5, 4, True, None), (8, 2, False, "block"), (8, 4, True, "block")]
    for N, d, causal, mk in cases:
        q, k, v, do = (r.standard_normal((1, 1, N, d)) for _ in range(4))
        scale = 1 / math.sqrt(d) * 1.3
        bm = None
        if mk:
            bm = np.array([[1, 0, 1, 0], [1, 1, 0, 0], [0, 1, 1, 0], [1, 0, 1, 1]], np.uint8)

        def phi(q_, k_, v_):
            o, _ = orc.forward(q_, k_, v_, scale, causal=causal, block_mask=bm, block=2)
            return float((o * do).sum())

        dq, dk, dv, _ = orc.backward(q, k, v, do, scale, causal=causal, block_mask=bm, block=2)
        h = 1e-6
        for which, g in ((0, dq), (1, dk), (2, dv)):
            fd = np.zeros_like(g)
            for idx in np.ndindex(g.shape):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][idx] += h
                args_m[which][idx] -= h
                fd[idx] = (phi(*args_p) - phi(*args_m)) / (2 * h)
            err = np.linalg.norm(fd - g) / max(np.linalg.norm(fd), 1e-30)
            assert err <= 1e-6, (N, d, causal, mk, which, err)


def pin_dvec(orc):
    """D_i = rowsum(P o dP) equals dO_i . O_i [P2 "Backward Pass of flashattention"]."""
    r = _rng(4)
    q, k, v, do = (r.standard_normal((1, 2, 33, 8)) for _ in range(4))
    for causal in (False, True):
        o, _ = orc.forward(q, k, v, 0.4, causal=causal)
        _, _, _, dvec = orc.backward(q, k, v, do, 0.4, causal=causal)
        np.testing.assert_allclose(dvec, (do * o).sum(axis=-1), atol=1e-12)


def pin_backward_rows(orc):
    r = _rng(6)
    q, k, v, do = (r.standard_normal((1, 2, 29, 4)) for _ in range(4))
    dq, dk, dv, _ = orc.backward(q, k, v, do, 0.5, causal=True)
    o, lse = orc.forward(q, k, v, 0.5, causal=True)
    rows = [0, 9, 28]
    np.testing.assert_allclose(orc.backward_rows_dq(q, k, v, do, 0.5, 0, 1, rows, causal=True),
                               dq[0, 1, rows], atol=1e-13)
    # row blocks partition the rows: their dK, dV contributions sum to the whole
    sdk, sdv = np.zeros_like(dk[0, 1]), np.zeros_like(dv[0, 1])
    for blk in (range(0, 10), range(10, 11), range(11, 29)):
        dqr, dkp, dvp, orr, lr = orc.backward_rows(q, k, v, do, 0.5, 0, 1, list(blk), causal=True)
        np.testing.assert_allclose(dqr, dq[0, 1, list(blk)], atol=1e-13)
        np.testing.assert_allclose(orr, o[0, 1, list(blk)], atol=1e-13)
        np.testing.assert_allclose(lr, lse[0, 1, list(blk)], atol=1e-13)
        sdk += dkp
        sdv += dvp
    np.testing.assert_allclose(sdk, dk[0, 1], atol=1e-12)
    np.testing.assert_allclose(sdv, dv[0, 1], atol=1e-12)
    # the same with dropout: the row blocks partition backward_dropout
    dq, dk, dv, _ = orc.backward_dropout(q, k, v, do, 0.5, 0.3, 77, causal=True)
    o, lse = orc.forward_dropout(q, k, v, 0.5, 0.3, 77, causal=True)
    sdk, sdv = np.zeros_like(dk[0, 1]), np.zeros_like(dv[0, 1])
    for blk in (range(0, 13), range(13, 29)):
        dqr, dkp, dvp, orr, lr = orc.backward_rows(q, k, v, do, 0.5, 0, 1, list(blk), causal=True,
                                                   dropout_p=0.3, seed=77)
        np.testing.assert_allclose(dqr, dq[0, 1, list(blk)], atol=1e-13)
        np.testing.assert_allclose(orr, o[0, 1, list(blk)], atol=1e-13)
        ofr, lfr = orc.forward_rows(q, k, v, 0.5, 0, 1, list(blk), causal=True, dropout_p=0.3, seed=77)
        np.testing.assert_allclose(ofr, o[0, 1, list(blk)], atol=1e-13)
        sdk += dkp
        sdv += dvp
    np.testing.assert_allclose(sdk, dk[0, 1], atol=1e-12)
    np.testing.assert_allclose(sdv, dv[0, 1], atol=1e-12)


# --------------------------------------------------------------------------- #
def pin_library(orc):
    """PyTorch's fp64 scaled_dot_product_attention and autograd, with masks
    built by torch ops, on shapes that span several blocks and a ragged tail."""
    r = _rng(5)
    B, H, N, d = 2, 3, 70, 16
    q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    bm = (r.random((5, 5)) < 0.4).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    bm[0, 3] = 1
    bm[3, 0] = 0                                           # make it asymmetric
    for causal, mask in ((False, None), (True, None), (False, bm), (True, bm)):
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        am = _dense_mask_torch(N, causal, mask, block=16)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am, scale=scale)
        ref.backward(torch.tensor(do))
        o, _ = orc.forward(q, k, v, scale, causal=causal, block_mask=mask, block=16)
        dq, dk, dv, _ = orc.backward(q, k, v, do, scale, causal=causal, block_mask=mask, block=16)
        np.testing.assert_allclose(o, ref.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def pin_block_masks(orc):
    """Sliding-window and dilated block masks against library routines
    (np.tril / np.triu band, np.eye, a parity checkerboard from np.indices),
    closed-form row counts, and attention-level special cases."""
    for N, left, right in ((1, 0, 0), (128, 0, 0), (129, 1, 0), (1000, 2, 1), (2048, 3, 5), (4096, 40, 40)):
        nb = -(-N // 128)
        band = np.triu(np.tril(np.ones((nb, nb), np.uint8), right), -left)
        np.testing.assert_array_equal(orc.window_block_mask(N, left, right), band)
    nb = 12
    N = nb * 128 - 5                                          # ragged last block
    np.testing.assert_array_equal(orc.window_block_mask(N, 0, 0), np.eye(nb, dtype=np.uint8))
    np.testing.assert_array_equal(orc.window_block_mask(N, nb, 0), np.tril(np.ones((nb, nb), np.uint8)))
    np.testing.assert_array_equal(orc.window_block_mask(N, 0, nb), np.triu(np.ones((nb, nb), np.uint8)))
    for w in (0, 1, 3):
        np.testing.assert_array_equal(orc.dilated_block_mask(N, w, 1), orc.window_block_mask(N, w, w))
        np.testing.assert_array_equal(orc.dilated_block_mask(N, w, 1, causal=True), orc.window_block_mask(N, w, 0))
    ii, jj = np.indices((nb, nb))
    np.testing.assert_array_equal(orc.dilated_block_mask(N, nb, 2), ((ii + jj) % 2 == 0).astype(np.uint8))
    nb2 = 64
    for w, r in ((1, 2), (3, 4), (2, 7)):
        m = orc.dilated_block_mask(nb2 * 128, w, r)
        mc = orc.dilated_block_mask(nb2 * 128, w, r, causal=True)
        np.testing.assert_array_equal(m, m.T)
        np.testing.assert_array_equal(mc, np.tril(m))
        interior = slice(w * r, nb2 - w * r)
        assert np.all(m[interior].sum(axis=1) == 2 * w + 1)
        assert np.all(mc[w * r:].sum(axis=1) == w + 1)
        i2, j2 = np.indices((nb2, nb2))
        assert np.all(m[i2 - j2 == r] == 1) and np.all(m[i2 - j2 == r + 1] == (1 if r == 1 else 0))
    # attention level: a causal window over every block is plain causal attention,
    # and a window of width 0 is causal attention inside each block independently
    r = _rng(11)
    blk, nbk = 8, 4
    N = blk * nbk - 3
    q, k, v = (r.standard_normal((1, 2, N, 4)) for _ in range(3))
    full = orc.window_block_mask(N, nbk, 0, block=blk)
    o_w, l_w = orc.forward(q, k, v, 0.5, causal=True, block_mask=full, block=blk)
    o_c, l_c = orc.forward(q, k, v, 0.5, causal=True)
    np.testing.assert_allclose(o_w, o_c, atol=1e-14)
    np.testing.assert_allclose(l_w, l_c, atol=1e-14)
    diag = orc.window_block_mask(N, 0, 0, block=blk)
    o_d, _ = orc.forward(q, k, v, 0.5, causal=True, block_mask=diag, block=blk)
    for b0 in range(0, N, blk):
        sl = slice(b0, min(N, b0 + blk))
        o_b, _ = orc.forward(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.5, causal=True)
        np.testing.assert_allclose(o_d[:, :, sl], o_b, atol=1e-14)


def pin_decode(orc):
    """Decoding against a key/value cache: the square causal case is the
    forward; one query token sees the whole cache either way; a short cache is
    the forward over its valid rows; PyTorch's fp64 attention with a
    bottom-right causal mask built by torch ops; rows with no visible key; and
    the split-KV merge equals the whole for every chunk size."""
    r = _rng(21)
    B, H, d = 2, 3, 8
    # square, causal: query i of N at position i
    N = 37
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    o, l = orc.decode(q, k, v, 0.4, causal=True)
    of, lf = orc.forward(q, k, v, 0.4, causal=True)
    np.testing.assert_allclose(o, of, atol=1e-13)
    np.testing.assert_allclose(l, lf, atol=1e-13)
    # one token: causal and non-causal agree
    q1 = r.standard_normal((B, H, 1, d))
    o1c, l1c = orc.decode(q1, k, v, 0.4, causal=True)
    o1, l1 = orc.decode(q1, k, v, 0.4)
    np.testing.assert_allclose(o1c, o1, atol=1e-14)
    np.testing.assert_allclose(l1c, l1, atol=1e-14)
    # a short cache: only its first L rows count
    seq = [11, 30]
    q4 = r.standard_normal((B, H, 4, d))
    o4, l4 = orc.decode(q4, k, v, 0.4, seqlens=seq)
    for b, L in enumerate(seq):
        ob, lb = orc.forward(q4[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.4)
        np.testing.assert_allclose(o4[b], ob[0], atol=1e-13)
        np.testing.assert_allclose(l4[b], lb[0], atol=1e-13)
    # library: torch SDPA with a bottom-right causal mask from torch.tril
    o4c, _ = orc.decode(q4, k, v, 0.4, seqlens=seq, causal=True)
    for b, L in enumerate(seq):
        am = torch.ones(4, L, dtype=torch.bool).tril(L - 4)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q4[b]), torch.tensor(k[b, :, :L]), torch.tensor(v[b, :, :L]), attn_mask=am, scale=0.4)
        np.testing.assert_allclose(o4c[b], ref.numpy(), atol=1e-13)
    # no visible key: a cache shorter than the query block, and an empty cache
    q6 = r.standard_normal((B, H, 6, d))
    o6, l6 = orc.decode(q6, k, v, 0.4, seqlens=[3, 0], causal=True)
    assert np.all(o6[0, :, :3] == 0) and np.all(np.isneginf(l6[0, :, :3]))   # positions -3..-1
    assert np.all(np.isfinite(l6[0, :, 3:]))
    assert np.all(o6[1] == 0) and np.all(np.isneginf(l6[1]))
    # the split-KV merge is exact for any chunk size
    for causal in (False, True):
        ow, lw = orc.decode(q6, k, v, 0.4, seqlens=[37, 9], causal=causal)
        for chunk in (1, 3, 8, 64):
            os_, ls_ = orc.decode_split(q6, k, v, 0.4, chunk, seqlens=[37, 9], causal=causal)
            np.testing.assert_allclose(os_, ow, atol=1e-13)
            np.testing.assert_allclose(ls_, lw, atol=1e-13)


def pin_philox(orc):
    """Philox4x32-10 against its published known-answer vectors, and the
    element-to-counter mapping of the dropout bytes against the same vectors:
    counter (j//4, i//4, h, b) and key (seed low, seed high) reproduce each
    vector's four output words as the 4 x 4 block of bytes (row i%4 = word,
    column j%4 = byte, little-endian)."""
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.json")) as f:
        kat = json.load(f)["vectors"]
    for vec in kat:
        ctr = np.array([int(x, 16) for x in vec["ctr"]], dtype=np.uint64)
        key = [int(x, 16) for x in vec["key"]]
        out = [int(x, 16) for x in vec["out"]]
        assert [int(x) for x in orc.philox4x32_10(ctr, key)] == out
        c0, c1, c2, c3 = (int(x) for x in ctr)
        seed = key[0] | (key[1] << 32)
        rows = 4 * c1 + np.arange(4)
        cols = 4 * c0 + np.arange(4)
        got = orc.dropout_bytes(c3, c2, rows, cols, seed)
        want = np.array([[(w >> (8 * j)) & 0xFF for j in range(4)] for w in out], dtype=np.uint8)
        np.testing.assert_array_equal(got, want)


def pin_dropout(orc):
    """Dropout: p = 0 is plain attention; keep rates and cross-head agreement
    match the binomial law; averaging over seeds gives the undropped output
    (unbiased); PyTorch autograd of softmax(S) o Z c V with the oracle's mask;
    central finite differences of the backward with a fixed mask."""
    r = _rng(31)
    B, H, N, d = 1, 2, 24, 4
    q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
    o0, l0 = orc.forward(q, k, v, 0.5, causal=True)
    od, ld = orc.forward_dropout(q, k, v, 0.5, 0.0, 7, causal=True)
    np.testing.assert_array_equal(od, o0)
    np.testing.assert_array_equal(ld, l0)
    g0 = orc.backward(q, k, v, do, 0.5, causal=True)
    gd = orc.backward_dropout(q, k, v, do, 0.5, 0.0, 7, causal=True)
    for a, b_ in zip(g0, gd):
        np.testing.assert_allclose(b_, a, atol=1e-14)
    assert orc.dropout_threshold(0.1) == 26 and orc.dropout_threshold(0.5) == 128
    # keep rate and independence (binomial bounds, 6 sigma)
    n = 256
    for pdrop in (0.1, 0.5):
        t = orc.dropout_threshold(pdrop)
        keep = 1 - t / 256
        z0 = orc.dropout_keep(0, 0, np.arange(n), np.arange(n), pdrop, 123)
        z1 = orc.dropout_keep(0, 1, np.arange(n), np.arange(n), pdrop, 123)
        z2 = orc.dropout_keep(1, 0, np.arange(n), np.arange(n), pdrop, 123)
        z3 = orc.dropout_keep(0, 0, np.arange(n), np.arange(n), pdrop, 124)
        m = n * n
        assert abs(z0.mean() - keep) <= 6 * math.sqrt(keep * (1 - keep) / m)
        agree = keep ** 2 + (1 - keep) ** 2
        for other in (z1, z2, z3, z0.T):
            assert abs((z0 == other).mean() - agree) <= 6 * math.sqrt(agree * (1 - agree) / m)
        # any sub-block is the same pairs' slice of the whole
        np.testing.assert_array_equal(orc.dropout_keep(0, 0, np.arange(5, 21), np.arange(3, 41), pdrop, 123),
                                      z0[5:21, 3:41])
    # unbiased: the mean over seeds approaches the undropped output
    acc = np.zeros_like(o0)
    S = 400
    for sd in range(S):
        acc += orc.forward_dropout(q, k, v, 0.5, 0.3, 1000 + sd, causal=True)[0]
    err = np.abs(acc / S - o0).max()
    assert err < 6 * np.abs(v).max() / math.sqrt(S), err
    # library: torch autograd of the dropped expression with the oracle's mask
    pdrop, seed = 0.25, 99
    c = 256.0 / (256 - orc.dropout_threshold(pdrop))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    z = torch.stack([torch.stack([torch.tensor(orc.dropout_keep(b_, h, np.arange(N), np.arange(N), pdrop, seed))
                                  for h in range(H)]) for b_ in range(B)])
    s_ = 0.5 * tq @ tk.transpose(-1, -2)
    s_ = s_.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    out = (torch.softmax(s_, dim=-1) * z * c) @ tv
    out.backward(torch.tensor(do))
    o_d, _ = orc.forward_dropout(q, k, v, 0.5, pdrop, seed, causal=True)
    dq, dk, dv, _ = orc.backward_dropout(q, k, v, do, 0.5, pdrop, seed, causal=True)
    np.testing.assert_allclose(o_d, out.detach().numpy(), atol=1e-13)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)
    # a head evaluated alone with its offsets equals that head of the whole
    full = orc.forward_dropout(q, k, v, 0.5, 0.3, 17)[0]
    alone = orc.forward_dropout(q[:, 1:2], k[:, 1:2], v[:, 1:2], 0.5, 0.3, 17, h0=1)[0]
    np.testing.assert_array_equal(alone[:, 0], full[:, 1])
    # finite differences with the mask fixed by the seed
    qs, ks, vs, dos = (x[:, :1, :9, :3].copy() for x in (q, k, v, do))
    g = orc.backward_dropout(qs, ks, vs, dos, 0.7, 0.4, 5)
    eps = 1e-6
    for idx, x in enumerate((qs, ks, vs)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            x[mi] += eps
            fp = (orc.forward_dropout(qs, ks, vs, 0.7, 0.4, 5)[0] * dos).sum()
            x[mi] -= 2 * eps
            fm = (orc.forward_dropout(qs, ks, vs, 0.7, 0.4, 5)[0] * dos).sum()
            x[mi] += eps
            num[mi] = (fp - fm) / (2 * eps)
        rel = np.linalg.norm(num - g[idx]) / max(np.linalg.norm(num), 1e-30)
        assert rel < 1e-6, (idx, rel)


def pin_fp8(orc):
    """8-bit inputs: e4m3 decoding against PyTorch's float8_e4m3fn for all 256
    codes and the format's landmarks; the 8-bit forward against PyTorch's fp64
    attention on the dequantised inputs; round-to-nearest e4m3 stays within a
    relative 2^-4; the error model's bound holds and its sigma matches the
    spread of randomly perturbed weights."""
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_decode(codes)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    np.testing.assert_array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    assert mine[0x38] == 1.0 and mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6
    assert mine[0xB8] == -1.0 and np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    # relative rounding error of e4m3 on its normal range
    r = _rng(41)
    x = np.exp2(r.uniform(-5.9, 8.7, 20000))
    xr = torch.tensor(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.max(np.abs(xr - x) / x) <= 2.0 ** -4
    # the 8-bit forward is attention on the dequantised inputs
    B, H, N, d = 1, 2, 40, 16
    q8, k8, v8 = (torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(s_)).mul(3).to(torch.float8_e4m3fn)
                  for s_ in (1, 2, 3))
    qd, kd, vd = (r.uniform(0.01, 0.5, (B, H)) for _ in range(3))
    u8 = [t.view(torch.uint8).numpy() for t in (q8, k8, v8)]
    o, lse, probs, vv = orc.forward_fp8(*u8, qd, kd, vd, 0.25, causal=True)
    tq, tk, tv = (t.to(torch.float64) * torch.tensor(s_)[..., None, None] for t, s_ in zip((q8, k8, v8), (qd, kd, vd)))
    am = torch.ones(N, N, dtype=torch.bool).tril()
    ref_o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am, scale=0.25).numpy()
    np.testing.assert_allclose(o, ref_o, atol=1e-13)
    # error model: worst case holds, sigma is the spread of random perturbations
    bound, sigma = orc.fp8_error_model(o, probs, vv)
    rel = 2.0 ** -4
    sq = np.zeros_like(o)
    S = 300
    for _ in range(S):
        w = probs * (1 + r.uniform(-rel, rel, probs.shape))
        do_ = np.einsum("bhij,bhjc->bhic", w, vv) - o
        assert np.all(np.abs(do_) <= bound + 1e-15)
        sq += do_ ** 2
    ratio = np.sqrt(sq.mean() / S) / np.sqrt((sigma ** 2).mean())
    assert 0.85 < ratio < 1.15, ratio


def pin_visibility(orc):
    """The visibility predicates against brute force on tiny shapes: key j is
    visible to query row i when j <= i under the causal mask [P2 causal
    masking] and when the block mask entry of (i // block, j // block) is set
    [P2 "Block-sparse Flashattention"]; a decoding query i of nq against a
    cache of L keys sits at position L - nq + i.  Covers row subsets, more keys
    than rows, ragged last blocks and the reduction of decoding with nq = L to
    the square causal mask."""
    r = _rng(29)
    for nq, nk, blk in ((1, 1, 4), (7, 7, 4), (9, 13, 4), (13, 9, 3), (16, 16, 8)):
        bm = (r.random((-(-nq // blk), -(-nk // blk))) < 0.5).astype(np.uint8)
        for causal in (False, True):
            for use_bm in (False, True):
                for rows in (None, np.array([nq - 1, 0, nq // 2])):
                    got = orc.visible(nq, nk, causal, bm if use_bm else None, blk, rows)
                    rr = range(nq) if rows is None else rows
                    want = np.zeros((len(rr), nk), dtype=bool)
                    for a, i in enumerate(rr):
                        for j in range(nk):
                            ok = (j <= i) if causal else True
                            if use_bm:
                                ok = ok and bool(bm[i // blk][j // blk])
                            want[a, j] = ok
                    np.testing.assert_array_equal(got, want)
    for nq, L in ((1, 1), (1, 5), (4, 4), (4, 11), (8, 9)):
        for causal in (False, True):
            want = np.array([[(not causal) or j <= L - nq + i for j in range(L)] for i in range(nq)])
            np.testing.assert_array_equal(orc.decode_visible(nq, L, causal), want)
    for L in (1, 6, 17):
        np.testing.assert_array_equal(orc.decode_visible(L, L, True), orc.visible(L, L, True))


def _bf16(x):
    """Round to bf16 (round to nearest even) and back, through PyTorch."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def pin_grad_error_model(orc):
    """The gradient error model against the rounding it describes: (1) a bf16
    pipeline simulated with real round-to-nearest-even bf16 values at every
    rounding point (forward P for P V, stored O, backward P for dV, dS, the
    outputs), with O normalised by the rounded or the exact row sum, stays
    inside u |r| + (1 + u)(6 sigma + acc) everywhere; (2) uniform relative
    perturbations of size u at those points spread with an RMS at most the
    model's sigma and not far below it (the model is an upper bound, not a
    vacuous one); (3) one wrong row of dQ or dK breaks the bound."""
    u = orc.BF16_U
    r = _rng(57)
    cases = [(1, 2, 160, 32, False, 1.0, None), (1, 1, 200, 64, True, 3.0, None),
             (1, 1, 256, 32, False, 1.0, np.array([[1, 0], [1, 1]], np.uint8))]
    for B, H, N, d, causal, amp, bm in cases:
        q, k, v, do = (_bf16(r.standard_normal((B, H, N, d)) * amp) for _ in range(4))
        s = 1 / math.sqrt(d)
        ref = orc.backward(q, k, v, do, s, causal=causal, block_mask=bm)[:3]
        sig, acc = orc.grad_error_model(q, k, v, do, s, causal=causal, block_mask=bm, row_chunk=64)
        vis = _dense_mask_torch(N, causal, bm).numpy()
        for rounded_sum in (True, False):
            sim = [np.zeros_like(q) for _ in range(3)]
            for b in range(B):
                for h in range(H):
                    qh, kh, vh, doh = q[b, h], k[b, h], v[b, h], do[b, h]
                    sc = np.where(vis, s * (qh @ kh.T), -np.inf)
                    f = np.exp(sc - sc.max(axis=1)[:, None])
                    fh = _bf16(f)
                    o = _bf16((fh @ vh) / (fh if rounded_sum else f).sum(axis=1)[:, None])
                    p = f / f.sum(axis=1)[:, None]
                    ds = _bf16(p * (doh @ vh.T - (doh * o).sum(axis=1)[:, None]))
                    sim[0][b, h] = _bf16(s * ds @ kh)
                    sim[1][b, h] = _bf16(s * ds.T @ qh)
                    sim[2][b, h] = _bf16(_bf16(p).T @ doh)
            for g, rr, sg, ac in zip(sim, ref, sig, acc):
                assert np.all(np.abs(g - rr) <= u * np.abs(rr) + (1 + u) * (6 * sg + ac))
        # planted wrong rows are caught
        for which in (0, 1):
            bad = ref[which].copy()
            bad[0, 0, [3, 4]] = bad[0, 0, [4, 3]]
            assert np.any(np.abs(bad - ref[which]) > u * np.abs(ref[which]) + (1 + u) * (6 * sig[which] + acc[which]))
        if amp == 1.0 and bm is None:
            for g, sg, ac in zip(ref, sig, acc):
                assert np.median((6 * sg + ac) / np.maximum(np.abs(g), 1e-30)) < 0.1
    # uniform perturbations of size u: RMS spread against the model's sigma
    B, H, N, d = 1, 1, 96, 16
    q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
    s = 0.25
    ref = orc.backward(q, k, v, do, s, causal=True)[:3]
    sig, _ = orc.grad_error_model(q, k, v, do, s, causal=True, f32=0.0)
    p = np.where(_dense_mask_torch(N, True).numpy(), np.exp(s * (q[0, 0] @ k[0, 0].T)), 0.0)
    p /= p.sum(axis=1)[:, None]
    sq = [np.zeros((N, d)) for _ in range(3)]
    S = 40
    for _ in range(S):
        w = p * (1 + r.uniform(-u, u, p.shape))
        o = (w @ v[0, 0]) / w.sum(axis=1)[:, None] * (1 + r.uniform(-u, u, (N, d)))
        dp = do[0, 0] @ v[0, 0].T
        ds = p * (dp - (do[0, 0] * o).sum(axis=1)[:, None]) * (1 + r.uniform(-u, u, p.shape))
        g = (s * ds @ k[0, 0], s * ds.T @ q[0, 0], (p * (1 + r.uniform(-u, u, p.shape))).T @ do[0, 0])
        for i in range(3):
            sq[i] += (g[i] - ref[i][0, 0]) ** 2
    for i in range(3):
        ratio = math.sqrt((sq[i] / S).mean()) / math.sqrt((sig[i] ** 2).mean())
        assert 0.4 < ratio < 1.1, (i, ratio)


def pin_forward_error_bound(orc):
    """The forward's P-rounding bound against the rounding it describes: a
    forward whose P V product takes round-to-nearest-even bf16 weights,
    normalised by the rounded or by the exact row sum, stays inside
    u ((P |V|) + |O|) everywhere, also on x3 inputs with peaked rows; on
    those rows the rounding alone exceeds 1e-2; and moving 1 % of a row's
    weight to another key breaks the bound."""
    u = orc.BF16_U
    r = _rng(61)
    seen_big = False
    for B, H, N, d, amp, causal in ((1, 2, 192, 64, 3.0, True), (1, 1, 256, 128, 1.0, False),
                                    (1, 1, 300, 64, 3.0, False)):
        q, k, v = (_bf16(r.standard_normal((B, H, N, d)) * amp) for _ in range(3))
        s = 1 / math.sqrt(d)
        o, _ = orc.forward(q, k, v, s, causal=causal)
        bound = orc.forward_error_bound(q, k, v, s, causal=causal, row_chunk=100)
        vis = _dense_mask_torch(N, causal).numpy()
        for b in range(B):
            for h in range(H):
                sc = np.where(vis, s * (q[b, h] @ k[b, h].T), -np.inf)
                f = np.exp(sc - sc.max(axis=1)[:, None])
                fh = _bf16(f)
                for den in (fh.sum(axis=1), f.sum(axis=1)):
                    err = np.abs((fh @ v[b, h]) / den[:, None] - o[b, h])
                    assert np.all(err <= bound[b, h] * (1 + 1e-6) + 1e-12)
                    seen_big |= bool(err.max() > 1e-2)
                # a wrong weight: 1 % of each row's mass moved to key 0
                p = f / f.sum(axis=1)[:, None]
                pw = 0.99 * p
                pw[:, 0] += 0.01
                err = np.abs(pw @ v[b, h] - o[b, h])
                assert np.any(err > bound[b, h])
    assert seen_big


ALL_PINS = [pin_worked_example, pin_closed_forms, pin_invariants, pin_backward_fd,
            pin_dvec, pin_backward_rows, pin_library, pin_block_masks, pin_decode, pin_philox, pin_dropout, pin_fp8,
            pin_visibility, pin_grad_error_model,
            pin_forward_error_bound]
