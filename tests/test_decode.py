"""Decoding against a key/value cache (split over the cache, chunks merged by
the statistics merge): the CUDA path against the fp64 oracle, element by
element, with the forward's tolerances (|O - O_ref| <= 1e-2 + 2^-8 |O_ref|,
LSE relative error <= 1e-3 relative to max(|LSE|, 1))."""
import math

import numpy as np
import pytest
import torch

from attn_fwd_gb300.inputs import make_decode_inputs
import oracle

pytestmark = pytest.mark.gpu

O_ATOL = 1e-2
BF16_HALF_ULP_REL = 2.0 ** -8
LSE_RTOL = 1e-3


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


def _check(o_gpu, lse_gpu, o_ref, lse_ref, what):
    o_gpu = o_gpu.float().cpu().numpy()
    lse_gpu = lse_gpu.float().cpu().numpy()
    assert np.isfinite(o_gpu).all(), what
    excess = (np.abs(o_gpu - o_ref) - (O_ATOL + BF16_HALF_ULP_REL * np.abs(o_ref))).max()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), what
    assert np.all(o_gpu[~fin] == 0), f"{what}: rows without visible keys must be 0"
    err_l = (np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1.0)).max() if fin.any() else 0.0
    assert excess <= 0, f"{what}: O error exceeds 1e-2 + 2^-8|O| by {excess}"
    assert err_l <= LSE_RTOL, f"{what}: LSE rel error {err_l}"


CASES = [
    # B, H, Nq, Nk, d, seqlens, causal
    (1, 1, 1, 1, 64, None, False),
    (1, 2, 1, 64, 128, None, True),            # one chunk: the split kernel writes O itself
    (1, 2, 1, 100, 128, None, False),
    (2, 4, 1, 1000, 64, [1000, 37], True),
    (2, 3, 4, 4096, 128, [4096, 4000], True),
    (1, 2, 8, 777, 128, None, True),
    (3, 2, 3, 5000, 64, [0, 1, 5000], True),   # empty cache; a cache shorter than the queries
    (2, 2, 5, 3000, 128, [2999, 65], False),
    (1, 8, 2, 65536, 128, None, False),        # hundreds of chunks
    (2, 16, 1, 32768, 128, [32768, 20001], True),
    # several tokens, two keys per lane: one tile (the second warp idle),
    # partial last tiles with both key groups, odd tile counts
    (1, 3, 4, 50, 128, None, True),
    (2, 2, 8, 200, 64, [200, 97], True),
    (1, 4, 6, 4133, 128, None, False),
    (2, 2, 7, 64, 128, [64, 33], True),
    (64, 64, 2, 96, 64, None, True),           # 4096 (batch, head) pairs, two tiles each
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,seqlens,causal", CASES)
def test_decode_matches_oracle(fa, B, H, Nq, Nk, d, seqlens, causal):
    t = make_decode_inputs(B, H, Nq, Nk, d, seed=Nk + Nq)
    scale = 1 / math.sqrt(d)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    sl = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    o, lse = fa.decode(q, k, v, seqlens_k=sl, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    ro, rl = oracle.decode(t["q"].double().numpy(), t["k"].double().numpy(), t["v"].double().numpy(), scale,
                           seqlens=seqlens, causal=causal)
    _check(o, lse, ro, rl, f"B={B} H={H} Nq={Nq} Nk={Nk} d={d} seqlens={seqlens} causal={causal}")


def test_decode_square_causal_equals_forward(fa):
    """The last 8 queries of a 128-token causal forward, decoded against the
    whole 128-row cache, give the same rows: both CUDA paths agree."""
    q = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    k = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    v = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    of, lf = fa.forward(qd, kd, vd, causal=True)
    od, ld = fa.decode(qd[:, :, 120:].contiguous(), kd, vd, causal=True)
    torch.cuda.synchronize()
    assert (of[:, :, 120:].float() - od.float()).abs().max().item() <= 2 * 2.0 ** -8 * of.float().abs().max().item() + 1e-2
    assert (lf[:, :, 120:] - ld).abs().max().item() <= 1e-3 * lf.abs().max().item()


def test_decode_outputs_stay_inside_their_rows(fa):
    B, H, Nq, Nk, d = 2, 3, 3, 2000, 128
    t = make_decode_inputs(B, H, Nq, Nk, d, seed=1)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    n, pad = B * H * Nq * d, 4096
    obuf = torch.full((n + pad,), 3.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * Nq + pad,), 3.0, dtype=torch.float32, device="cuda")
    o, lse = obuf[:n].view(B, H, Nq, d), lbuf[:B * H * Nq].view(B, H, Nq)
    nws = fa.fa_decode_workspace_bytes(B, H, Nq, Nk, d)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda") if nws else None
    fa.fa_decode(q, k, v, o, lse, None, 1 / math.sqrt(d), causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    assert torch.all(obuf[n:] == 3.0) and torch.all(lbuf[B * H * Nq:] == 3.0)
