"""Comparisons of the CUDA path's outputs with the fp64 oracle, shared by the
GPU parity tests.

Forward: |O - O_ref| <= 1e-2 + 2^-8 |O_ref| element-wise (the stated 1e-2
beyond the bf16 rounding of O itself), LSE relative error <= 1e-3 against
max(|LSE|, 1).  Gradients: relative L2 <= 2e-2 per tensor of each head and per
128-row tile (reference norm floored at an RMS of 1e-3), and every element
inside the oracle's gradient error model, |g - r| <= u |r| + (1 + u)(6 sigma +
acc).
"""
import numpy as np
import torch

import oracle

O_ATOL = 1e-2
BF16_HALF_ULP_REL = 2.0 ** -8
LSE_RTOL = 1e-3
GRAD_RTOL = 2e-2
GRAD_SIGMAS = 6
TILE = 128


def dev(t):
    return t.to("cuda")


def np64(t):
    return t.double().numpy()


def check_fwd(o_gpu, lse_gpu, o_ref, lse_ref, what="", pbound=None):
    """O within 1e-2 + 2^-8 |O_ref| (+ pbound: the oracle's bound on the
    effect of bf16 probabilities in P V, used on inputs of amplitude > 1,
    where that rounding alone can exceed 1e-2); LSE relative 1e-3."""
    o_gpu = o_gpu.float().cpu().numpy()
    lse_gpu = lse_gpu.float().cpu().numpy()
    assert np.isfinite(o_gpu).all(), what
    err_o = np.abs(o_gpu - o_ref).max()
    limit = O_ATOL + BF16_HALF_ULP_REL * np.abs(o_ref) + (0.0 if pbound is None else pbound)
    excess = (np.abs(o_gpu - o_ref) - limit).max()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), what
    err_l = (np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1.0)).max() if fin.any() else 0.0
    assert excess <= 0, f"{what}: O error {err_o} exceeds its bound by {excess}"
    assert err_l <= LSE_RTOL, f"{what}: LSE rel error {err_l}"
    return err_o, err_l


def np32(g):
    return g.float().cpu().numpy() if torch.is_tensor(g) else np.asarray(g)


def rel_l2(g, r):
    """Relative L2 error; the reference norm is floored at an RMS of 1e-3 so that
    an exactly vanishing gradient (one key: dS = P (dP - D) = 0) compares its
    rounding noise against an absolute scale instead of against zero."""
    g = np32(g)
    return np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-3 * np.sqrt(r.size))


def tile_rel_l2(g, r):
    """The largest relative L2 error over the 128-row tiles of every head
    (rows on the second-to-last axis; the last tile may be shorter)."""
    g = np32(g)
    n = r.shape[-2]
    gh = g.reshape(-1, n, r.shape[-1])
    rh = r.reshape(-1, n, r.shape[-1])
    worst = 0.0
    for t0 in range(0, n, TILE):
        a, b = gh[:, t0:t0 + TILE], rh[:, t0:t0 + TILE]
        err = np.sqrt(((a - b) ** 2).sum(axis=(1, 2)))
        ref = np.maximum(np.sqrt((b ** 2).sum(axis=(1, 2))), 1e-3 * np.sqrt(b[0].size))
        worst = max(worst, float((err / ref).max()))
    return worst


def grad_excess(g, r, sig, acc):
    """Largest |g - r| beyond u |r| + (1 + u)(6 sigma + acc): <= 0 when every
    element is inside the gradient error model's bound."""
    u = oracle.BF16_U
    g = np32(g)
    return float((np.abs(g - r) - (u * np.abs(r) + (1 + u) * (GRAD_SIGMAS * sig + acc))).max())


def check_device_status(fa):
    torch.cuda.synchronize()
    rc = fa.fa_get_device_error()
    assert rc == 0, fa.status_string(rc)


def check_bwd(g, ref, what, model=None):
    """Per tensor and per 128-row tile relative L2 <= 2e-2; with the error
    model (sigma, acc) of the same heads, every element inside its bound."""
    for i, (name, a, r) in enumerate(zip(("dQ", "dK", "dV"), g, ref)):
        assert torch.isfinite(a).all(), f"{what}: {name} not finite"
        rel = rel_l2(a, r)
        assert rel <= GRAD_RTOL, f"{what}: {name} rel-L2 error {rel}"
        trel = tile_rel_l2(a, r)
        assert trel <= GRAD_RTOL, f"{what}: {name} worst 128-row tile rel-L2 error {trel}"
        if model is not None:
            ex = grad_excess(a, r, model[0][i], model[1][i])
            assert ex <= 0, f"{what}: {name} exceeds the element bound by {ex}"


def oracle_bwd(f64, scale, causal=False, bm=None):
    """The oracle's dQ, dK, dV of whole heads and their error model."""
    ref = oracle.backward(f64["q"], f64["k"], f64["v"], f64["do"], scale, causal=causal, block_mask=bm)[:3]
    model = oracle.grad_error_model(f64["q"], f64["k"], f64["v"], f64["do"], scale, causal=causal, block_mask=bm)
    return ref, model
