"""Seeded random configurations, forward and backward against the fp64 oracle
element by element: batch, heads, sequence length (ragged), head dimension,
mask kind (none, causal, random block mask, block mask with the causal flag,
sliding window) and dropout drawn from one fixed generator, so every run
checks the same 24 cases.  Tolerances as in the other parity tests: O within
1e-2 + 2^-8 |O|, LSE relative 1e-3 (against max(|LSE|, 1)), gradients
relative L2 2e-2 per tensor and per 128-row tile (reference norm floored at an
RMS of 1e-3) and, without dropout, every element inside the oracle's gradient
error model.
"""
import math

import numpy as np
import pytest
import torch

from attn_fwd_gb300.inputs import make_qkvdo
import oracle
from tests.parity_checks import check_bwd, oracle_bwd

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=20261202):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(r.integers(1, 3))
        H = int(r.integers(1, 4))
        N = int(r.integers(1, 1601))
        d = int(r.choice([64, 128]))
        mask = str(r.choice(["none", "causal", "block", "block_causal", "window"]))
        drop = float(r.choice([0.0, 0.0, 0.0, 0.1, 0.3]))
        out.append((i, B, H, N, d, mask, drop))
    return out


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


def _mask(N, kind, seed):
    nb = (N + 127) // 128
    if kind in ("block", "block_causal"):
        g = torch.Generator().manual_seed(seed)
        bm = (torch.rand((nb, nb), generator=g) < 0.35).to(torch.uint8)
        bm.fill_diagonal_(1)
        return bm
    if kind == "window":
        return torch.from_numpy(oracle.window_block_mask(N, 2, 1).astype(np.uint8))
    return None


@pytest.mark.parametrize("i,B,H,N,d,mask,drop", _cases())
def test_random_configuration(fa, i, B, H, N, d, mask, drop):
    what = f"case {i}: B{B} H{H} N{N} d{d} mask={mask} dropout={drop}"
    t = make_qkvdo(B, H, N, d, seed=500 + i)
    scale = 1 / math.sqrt(d)
    causal = mask in ("causal", "block_causal")
    bm = _mask(N, mask, 900 + i)
    seed = 77 + i
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    bmd = None if bm is None else bm.cuda()
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=bmd, dropout_p=drop, seed=seed)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=bmd, dropout_p=drop,
                             seed=seed)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0, what
    f64 = {n: t[n].double().numpy() for n in ("q", "k", "v", "do")}
    bmn = None if bm is None else bm.numpy()
    model = None
    if drop:
        ro, rl = oracle.forward_dropout(f64["q"], f64["k"], f64["v"], scale, drop, seed, causal=causal,
                                        block_mask=bmn)
        ref = oracle.backward_dropout(f64["q"], f64["k"], f64["v"], f64["do"], scale, drop, seed, causal=causal,
                                      block_mask=bmn)[:3]
    else:
        ro, rl = oracle.forward(f64["q"], f64["k"], f64["v"], scale, causal=causal, block_mask=bmn)
        ref, model = oracle_bwd(f64, scale, causal, bmn)
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(og).all(), what
    excess = (np.abs(og - ro) - (1e-2 + 2.0 ** -8 * np.abs(ro))).max()
    assert excess <= 0, f"{what}: O error exceeds the bound by {excess}"
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lg), fin), what
    if fin.any():
        lerr = (np.abs(lg[fin] - rl[fin]) / np.maximum(np.abs(rl[fin]), 1.0)).max()
        assert lerr <= 1e-3, f"{what}: LSE rel error {lerr}"
    check_bwd((dq, dk, dv), ref, what, model)
