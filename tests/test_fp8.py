"""The 8-bit (e4m3) forward against the fp64 oracle on the same e4m3 inputs:
exact attention on the dequantised inputs.  The kernel rounds P to e4m3
(3 mantissa bits), so the bound per element is the oracle's error model
(worst case over relative weight errors up to 2^-4) plus O's bf16 rounding; and the RMS error must stay within twice the standard
deviation of independent round-to-nearest errors, which a misplaced weight
would exceed by far."""
import math

import numpy as np
import pytest
import torch

from attn_fwd_gb300.inputs import make_fp8_inputs
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


def _run(fa, t, causal, scale):
    dev = {n: t[n].cuda() for n in t}
    o, lse = fa.forward_fp8(dev["q8"], dev["k8"], dev["v8"], dev["qd"], dev["kd"], dev["vd"], causal=causal,
                            scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _check(o, lse, t, causal, scale, what):
    u8 = [t[n].view(torch.uint8).numpy() for n in ("q8", "k8", "v8")]
    ro, rl, probs, v = oracle.forward_fp8(*u8, t["qd"].double().numpy(), t["kd"].double().numpy(),
                                          t["vd"].double().numpy(), scale, causal=causal)
    bound, sigma = oracle.fp8_error_model(ro, probs, v)
    err = np.abs(o - ro)
    limit = bound + 2.0 ** -8 * np.abs(ro) + 1e-3
    assert np.isfinite(o).all(), what
    assert (err <= limit).all(), f"{what}: worst excess {(err - limit).max()}"
    rms_err = np.sqrt((err ** 2).mean())
    rms_expect = np.sqrt((sigma ** 2 + (2.0 ** -8 * ro) ** 2 / 3).mean())
    assert rms_err <= 2 * rms_expect, f"{what}: RMS error {rms_err} vs expected {rms_expect}"
    lerr = (np.abs(lse - rl) / np.maximum(np.abs(rl), 1.0)).max()
    assert lerr <= 1e-3, f"{what}: LSE rel error {lerr}"


CASES = [
    # B, H, N, causal
    (1, 2, 256, False),
    (1, 2, 384, True),
    (2, 1, 200, True),
    (1, 1, 1000, False),
    (1, 2, 1024, True),
    (2, 2, 129, False),
]


@pytest.mark.parametrize("B,H,N,causal", CASES)
def test_fp8_forward_matches_oracle(fa, B, H, N, causal):
    t = make_fp8_inputs(B, H, N, 128, seed=N)
    scale = 1 / math.sqrt(128)
    o, lse = _run(fa, t, causal, scale)
    _check(o, lse, t, causal, scale, f"B={B} H={H} N={N} causal={causal}")


def test_fp8_forward_long_sampled_head(fa):
    """B2 H16 N4096 causal: two whole heads through the oracle."""
    B, H, N = 2, 16, 4096
    t = make_fp8_inputs(B, H, N, 128, seed=4096)
    scale = 1 / math.sqrt(128)
    o, lse = _run(fa, t, True, scale)
    for b, h in ((0, 3), (1, 15)):
        th = {n: t[n][b:b + 1, h:h + 1].contiguous() for n in t}
        _check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], th, True, scale, f"N=4096 head ({b}, {h})")


def test_fp8_forward_persistent_odd_tiles(fa):
    """B4 H16 N1100 causal: 320 query-tile pairs (more than SMs) whose last pair
    per head has one tile; whole heads through the oracle, every head finite."""
    B, H, N = 4, 16, 1100
    t = make_fp8_inputs(B, H, N, 128, seed=1100)
    scale = 1 / math.sqrt(128)
    o, lse = _run(fa, t, True, scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    for b, h in ((0, 0), (2, 7), (3, 15)):
        th = {n: t[n][b:b + 1, h:h + 1].contiguous() for n in t}
        _check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], th, True, scale, f"N=1100 head ({b}, {h})")


def test_fp8_outputs_stay_inside_their_rows(fa):
    B, H, N, d = 1, 2, 300, 128
    t = make_fp8_inputs(B, H, N, d, seed=3)
    dev = {n: t[n].cuda() for n in t}
    n, pad = B * H * N * d, 4096
    obuf = torch.full((n + pad,), 3.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * N + pad,), 3.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fa_fwd_fp8(dev["q8"], dev["k8"], dev["v8"], obuf[:n].view(B, H, N, d), lbuf[:B * H * N].view(B, H, N),
                  dev["qd"], dev["kd"], dev["vd"], 1 / math.sqrt(d), True, ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    assert torch.all(obuf[n:] == 3.0) and torch.all(lbuf[B * H * N:] == 3.0)
