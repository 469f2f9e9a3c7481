"""fa_fwd_bwd_host (host tensors streamed through the device in chunks of
heads) against the device-resident calls on the same inputs: the same kernels
on the same per-head data, so O, LSE, dK and dV agree bit for bit; dQ is
summed with fp32 atomics in an order that may differ, so it agrees to within
the rounding of one bf16 step."""
import math

import pytest
import torch

from attn_fwd_gb300.inputs import make_qkvdo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


CASES = [
    # B, H, N, d, causal, block-mask density (None: no block mask); chunks
    (2, 16, 1024, 128, True, None),       # one chunk (two waves need 38 heads)
    (2, 16, 4096, 128, True, None),       # chunks of 4, 8, 8, 8, 4 heads
    (1, 27, 4096, 64, False, 0.3),        # chunks of 5, 9, 9, 4 heads, block mask
    (3, 25, 2048, 128, True, None),       # chunks of 10, 19, 19, 19, 8 heads
    (1, 3, 1000, 64, True, 0.5),          # one chunk, ragged N, block mask and causal
]


@pytest.mark.parametrize("B,H,N,d,causal,density", CASES)
def test_host_streamed_matches_device_calls(fa, B, H, N, d, causal, density):
    t = make_qkvdo(B, H, N, d, seed=N + H)
    scale = 1 / math.sqrt(d)
    bm = None
    if density is not None:
        nb = -(-N // 128)
        g = torch.Generator().manual_seed(N)
        m = (torch.rand((nb, nb), generator=g) < density).to(torch.uint8)
        m.fill_diagonal_(1)
        bm = m.cuda()
    host = {n: t[n].pin_memory() for n in ("q", "k", "v", "do")}
    o_h, lse_h, dq_h, dk_h, dv_h = fa.forward_backward_host(host["q"], host["k"], host["v"], host["do"],
                                                             causal=causal, scale=scale, block_mask=bm)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    dev = {n: t[n].cuda() for n in ("q", "k", "v", "do")}
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], causal=causal, scale=scale, block_mask=bm)
    dq, dk, dv = fa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], causal=causal, scale=scale,
                             block_mask=bm)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o.cpu())
    assert torch.equal(lse_h, lse.cpu())
    assert torch.equal(dk_h, dk.cpu())
    assert torch.equal(dv_h, dv.cpu())
    torch.testing.assert_close(dq_h.float(), dq.cpu().float(), rtol=2 ** -7, atol=1e-4)


def test_host_streamed_back_to_back_calls_reuse_the_workspace(fa):
    """Two calls in a row on one workspace (the second's chunks reuse buffer
    sets the first just copied out of) give the same results."""
    B, H, N, d = 1, 20, 2048, 128
    t = make_qkvdo(B, H, N, d, seed=7)
    host = {n: t[n].pin_memory() for n in ("q", "k", "v", "do")}
    ws = torch.empty(fa.fa_fwd_bwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    r1 = fa.forward_backward_host(host["q"], host["k"], host["v"], host["do"], causal=True, ws=ws)
    r2 = fa.forward_backward_host(host["q"], host["k"], host["v"], host["do"], causal=True, ws=ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), r1, r2):
        if name == "dq":
            torch.testing.assert_close(a.float(), b.float(), rtol=2 ** -7, atol=1e-4)
        else:
            assert torch.equal(a, b), name


FWD_CASES = [
    # B, H, N, d, causal, block-mask density (None: no block mask)
    (1, 32, 4096, 128, True, None),       # 16 CTAs a head: chunks of 8, 16, 8 heads
    (2, 8, 2048, 64, False, 0.4),         # one chunk, block mask
    (1, 5, 1000, 128, True, None),        # one chunk, ragged N
]


@pytest.mark.parametrize("B,H,N,d,causal,density", FWD_CASES)
def test_host_streamed_forward_matches_device_call(fa, B, H, N, d, causal, density):
    t = make_qkvdo(B, H, N, d, seed=N + 3 * H, with_dout=False)
    scale = 1 / math.sqrt(d)
    bm = None
    if density is not None:
        nb = -(-N // 128)
        g = torch.Generator().manual_seed(N + 1)
        m = (torch.rand((nb, nb), generator=g) < density).to(torch.uint8)
        m.fill_diagonal_(1)
        bm = m.cuda()
    host = {n: t[n].pin_memory() for n in ("q", "k", "v")}
    o_h, lse_h = fa.forward_host(host["q"], host["k"], host["v"], causal=causal, scale=scale, block_mask=bm)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    o, lse = fa.forward(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), causal=causal, scale=scale, block_mask=bm)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o.cpu())
    assert torch.equal(lse_h, lse.cpu())
