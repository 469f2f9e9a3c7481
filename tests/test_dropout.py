"""Dropout with regenerated masks: the CUDA path against the fp64 oracle
(forward_dropout / backward_dropout, the same Philox4x32-10 mask definition
implemented independently on both sides), element by element, with the
forward's and backward's tolerances."""
import math

import numpy as np
import pytest
import torch

from attn_fwd_gb300.inputs import make_qkvdo
import oracle

pytestmark = pytest.mark.gpu

O_ATOL, BF16_HALF_ULP_REL, LSE_RTOL, GRAD_RTOL = 1e-2, 2.0 ** -8, 1e-3, 2e-2


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


def _check_fwd(o, lse, ro, rl, what):
    o, lse = o.float().cpu().numpy(), lse.float().cpu().numpy()
    assert np.isfinite(o).all(), what
    excess = (np.abs(o - ro) - (O_ATOL + BF16_HALF_ULP_REL * np.abs(ro))).max()
    assert excess <= 0, f"{what}: O error exceeds the bound by {excess}"
    err_l = (np.abs(lse - rl) / np.maximum(np.abs(rl), 1.0)).max()
    assert err_l <= LSE_RTOL, f"{what}: LSE rel error {err_l}"


def _rel_l2(g, r):
    g = g.float().cpu().numpy()
    return np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-3 * np.sqrt(r.size))


CASES = [
    # B, H, N, d, causal, p, seed, block-mask keep probability
    (1, 2, 256, 64, False, 0.1, 1, None),
    (1, 2, 384, 128, True, 0.3, 2 ** 40 + 7, None),
    (2, 1, 200, 64, True, 0.5, 3, None),
    (1, 1, 512, 128, False, 0.2, 0xDEADBEEFCAFEF00D, 0.5),
    (1, 2, 1000, 128, True, 0.1, 5, None),
    (1, 1, 640, 64, True, 0.25, 6, 0.6),
    # sliding windows: the two query tiles of a CTA share all but one key
    # tile, so the forward runs its shared-first round order
    (1, 2, 2048, 128, True, 0.2, 11, ("window", 3, 0)),
    (1, 1, 1500, 64, False, 0.15, 12, ("window", 2, 2)),
]


def _mask(N, keep_p, seed):
    if keep_p is None:
        return None
    if isinstance(keep_p, tuple):
        return torch.from_numpy(oracle.window_block_mask(N, keep_p[1], keep_p[2]).astype(np.uint8))
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((nb, nb), generator=g) < keep_p).to(torch.uint8)
    bm.fill_diagonal_(1)
    return bm


@pytest.mark.parametrize("B,H,N,d,causal,p,seed,keep_p", CASES)
def test_dropout_matches_oracle(fa, B, H, N, d, causal, p, seed, keep_p):
    t = make_qkvdo(B, H, N, d, seed=N + d)
    scale = 1 / math.sqrt(d)
    bm = _mask(N, keep_p, N)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    bmd = None if bm is None else bm.cuda()
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=bmd, dropout_p=p, seed=seed)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=bmd, dropout_p=p, seed=seed)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    f64 = {n: t[n].double().numpy() for n in ("q", "k", "v", "do")}
    bmn = None if bm is None else bm.numpy()
    what = f"B={B} H={H} N={N} d={d} causal={causal} p={p}"
    ro, rl = oracle.forward_dropout(f64["q"], f64["k"], f64["v"], scale, p, seed, causal=causal, block_mask=bmn)
    _check_fwd(o, lse, ro, rl, what)
    ref = oracle.backward_dropout(f64["q"], f64["k"], f64["v"], f64["do"], scale, p, seed, causal=causal,
                                  block_mask=bmn)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref[:3]):
        err = _rel_l2(g, r)
        assert err <= GRAD_RTOL, f"{what}: {name} rel-L2 {err}"


def test_dropout_is_a_function_of_the_seed(fa):
    t = make_qkvdo(1, 2, 512, 128, seed=11)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o1, l1 = fa.forward(q, k, v, causal=True, dropout_p=0.2, seed=42)
    o2, l2 = fa.forward(q, k, v, causal=True, dropout_p=0.2, seed=42)
    o3, _ = fa.forward(q, k, v, causal=True, dropout_p=0.2, seed=43)
    g1 = fa.backward(q, k, v, o1, l1, do, causal=True, dropout_p=0.2, seed=42)
    g2 = fa.backward(q, k, v, o1, l1, do, causal=True, dropout_p=0.2, seed=42)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert not torch.equal(o1, o3)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])   # dK, dV: no atomics


def test_tiny_dropout_probability_is_plain_attention(fa):
    """p below 1/512 rounds to a zero byte threshold: nothing is dropped."""
    t = make_qkvdo(1, 1, 256, 64, seed=12)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=True, dropout_p=0.001, seed=1)
    o2, l2 = fa.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_dropout_long_sequence_sampled_head(fa):
    """B2 H16 N2048 d128 causal, p = 0.1: one head through the oracle."""
    B, H, N, d = 2, 16, 2048, 128
    t = make_qkvdo(B, H, N, d, seed=13)
    scale = 1 / math.sqrt(d)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, dropout_p=0.1, seed=2024)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, dropout_p=0.1, seed=2024)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    b, h = 1, 9
    sl = (slice(b, b + 1), slice(h, h + 1))
    f64 = {n: t[n][sl].double().numpy() for n in ("q", "k", "v", "do")}
    ro, rl = oracle.forward_dropout(f64["q"], f64["k"], f64["v"], scale, 0.1, 2024, causal=True, b0=b, h0=h)
    _check_fwd(o[b, h], lse[b, h], ro[0, 0], rl[0, 0], "N=2048 head (1, 9)")
    ref = oracle.backward_dropout(f64["q"], f64["k"], f64["v"], f64["do"], scale, 0.1, 2024, causal=True, b0=b, h0=h)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq[b, h], dk[b, h], dv[b, h]), ref[:3]):
        err = _rel_l2(g, r[0, 0])
        assert err <= GRAD_RTOL, f"N=2048 head (1, 9): {name} rel-L2 {err}"
