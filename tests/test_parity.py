"""CUDA path vs the fp64 oracle, element by element, on the same seeded inputs.

Tolerances (bf16 inputs, fp32 accumulation): forward O max-abs error <= 1e-2
beyond the rounding of O to bf16 itself (|O - O_ref| <= 1e-2 + 2^-8 |O_ref|:
2^-8 |x| is half a bf16 ulp, which alone exceeds 1e-2 once |O| > 2.56, as in
the x3-amplitude workload); LSE relative error <= 1e-3, relative to
max(|LSE|, 1).  Gradients dQ, dK, dV: relative L2 error <= 2e-2 for each
tensor of each head and for each 128-row tile of it (a wrong row moves a
tile's error by about 1/sqrt(128) = 9 %), the reference norm floored at an
RMS of 1e-3; and, where the whole head goes through the oracle, every element
within |g - r| <= u |r| + (1 + u)(6 sigma + acc): u = 2^-8 the output's own
rounding, sigma the propagated bf16 rounding of P, dS and O and acc the fp32
accumulation bound of the oracle's gradient error model.
Workloads the oracle cannot finish in seconds are checked on whole heads
through the oracle (every head of the N = 4096 and N = 8192 workloads, eight
of the N = 16384 one) and on sampled query rows.
"""
import math

import numpy as np
import pytest
import torch

from attn_fwd_gb300.inputs import WORKLOADS, make_block_mask, make_qkvdo, make_workload_inputs
import oracle
from tests.parity_checks import (GRAD_RTOL, check_bwd, check_device_status, check_fwd, dev, np64,
                                 oracle_bwd, rel_l2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import attn_fwd_gb300.fa as fa
    fa.load()
    fa.fa_set_wait_timeout_ns(500_000_000)   # a broken pipeline fails fast instead of waiting 2 s per CTA
    return fa


# --------------------------------------------------------------------------- #
# forward, oracle on every element
# --------------------------------------------------------------------------- #
SMALL = [
    # B, H, N, d, causal, mask_p
    (1, 1, 128, 64, False, None),
    (1, 1, 128, 128, True, None),
    (2, 3, 256, 64, True, None),
    (1, 2, 384, 128, False, None),       # odd tile count: the last CTA has one query tile
    (1, 2, 384, 64, True, None),
    (2, 1, 640, 128, True, None),
    (1, 2, 512, 64, False, 0.3),
    (1, 2, 768, 128, False, 0.25),
]


@pytest.mark.parametrize("B,H,N,d,causal,p", SMALL)
def test_forward_small(fa, B, H, N, d, causal, p):
    t = make_qkvdo(B, H, N, d, seed=10 + N + d, with_dout=False)
    scale = 1 / math.sqrt(d)
    bm = make_block_mask(N, seed=N, p=p) if p is not None else None
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]), causal=causal, scale=scale,
                        block_mask=None if bm is None else dev(bm))
    check_device_status(fa)
    ro, rl = oracle.forward(np64(t["q"]), np64(t["k"]), np64(t["v"]), scale, causal=causal,
                            block_mask=None if bm is None else bm.numpy())
    check_fwd(o, lse, ro, rl, f"B{B} H{H} N{N} d{d} causal={causal} p={p}")


def test_forward_workload_small_tile(fa):
    """The single-tile latency workload: B1 H1 N128 d64, seed 0."""
    w = WORKLOADS["fwd_b1h1n128d64"]
    t = make_workload_inputs(w)
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]), causal=w.causal, scale=w.scale)
    check_device_status(fa)
    ro, rl = oracle.forward(np64(t["q"]), np64(t["k"]), np64(t["v"]), w.scale)
    check_fwd(o, lse, ro, rl, w.name)


def test_forward_workload_n1024(fa):
    w = WORKLOADS["fwdbwd_b4h8n1024d64"]
    t = make_workload_inputs(w)
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]), causal=w.causal, scale=w.scale)
    check_device_status(fa)
    ro, rl = oracle.forward(np64(t["q"]), np64(t["k"]), np64(t["v"]), w.scale)
    check_fwd(o, lse, ro, rl, w.name)


def test_forward_fully_masked_rows(fa):
    """Query blocks whose every block-mask byte is 0 get O = 0 and LSE = -inf."""
    B, H, N, d = 1, 2, 512, 64
    t = make_qkvdo(B, H, N, d, seed=77, with_dout=False)
    bm = torch.ones(4, 4, dtype=torch.uint8)
    bm[1, :] = 0
    bm[3, 1:] = 0
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]), block_mask=dev(bm))
    check_device_status(fa)
    ro, rl = oracle.forward(np64(t["q"]), np64(t["k"]), np64(t["v"]), 1 / 8, block_mask=bm.numpy())
    check_fwd(o, lse, ro, rl, "fully masked rows")
    assert torch.all(o[:, :, 128:256] == 0)


def test_forward_guard_bands(fa):
    """Outputs written through views of larger buffers leave the padding untouched."""
    B, H, N, d = 1, 2, 256, 128
    t = make_qkvdo(B, H, N, d, seed=5, with_dout=False)
    n = B * H * N * d
    pad = 4096
    obuf = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + n].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd(dev(t["q"]), dev(t["k"]), dev(t["v"]), o, lse, 1 / math.sqrt(d), causal=True)
    check_device_status(fa)
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[pad + n:] == 7.0)
    assert torch.all(lbuf[:pad] == 7.0) and torch.all(lbuf[pad + B * H * N:] == 7.0)


def test_forward_deterministic(fa):
    t = make_qkvdo(1, 4, 1024, 128, seed=6, with_dout=False)
    q, k, v = (dev(t[n]) for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k, v, causal=True)
    check_device_status(fa)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_forward_on_side_stream(fa):
    t = make_qkvdo(1, 2, 256, 64, seed=8, with_dout=False)
    q, k, v = (dev(t[n]) for n in ("q", "k", "v"))
    ref_o, ref_l = fa.forward(q, k, v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o, lse = fa.forward(q, k, v)
    s.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


# --------------------------------------------------------------------------- #
# forward at full workload sizes, sampled
# --------------------------------------------------------------------------- #
def _sampled_heads(BH, k, seed):
    r = np.random.default_rng(seed)
    return sorted(r.choice(BH, size=min(k, BH), replace=False).tolist())


@pytest.mark.parametrize("name", ["fwdbwd_b2h16n4096d128_causal", "fwdbwd_b1h16n8192d128_blocksparse"])
def test_forward_workload_all_heads(fa, name):
    w = WORKLOADS[name]
    t = make_workload_inputs(w)
    bm = t.get("block_mask")
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]), causal=w.causal, scale=w.scale,
                        block_mask=None if bm is None else dev(bm))
    check_device_status(fa)
    o, lse = o.cpu(), lse.cpu()
    for hh in range(w.B * w.H):
        b, h = divmod(hh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rl = oracle.forward(np64(t["q"][sl]), np64(t["k"][sl]), np64(t["v"][sl]), w.scale,
                                causal=w.causal, block_mask=None if bm is None else bm.numpy())
        check_fwd(o[sl], lse[sl], ro, rl, f"{name} head {hh}")


PERSISTENT = [
    # B, H, N, d, causal: more query-tile pairs than SMs, so the forward's
    # persistent CTAs each walk several; ragged N, and an odd tile count whose
    # last pair of every head has one tile (its Q phase completes empty)
    (2, 16, 2000, 128, True),
    (4, 16, 1100, 64, False),
    (8, 8, 1100, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", PERSISTENT)
def test_forward_persistent_items(fa, B, H, N, d, causal):
    """Every (batch, head) of a multi-item persistent launch written once and
    right: all heads finite, sampled heads element by element."""
    n_items = (N + 255) // 256 * B * H
    assert n_items > 152
    t = make_qkvdo(B, H, N, d, seed=80 + N, with_dout=False)
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]), causal=causal, scale=scale)
    check_device_status(fa)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    for hh in sorted(set([0, B * H - 1] + _sampled_heads(B * H, 3, seed=N))):
        b, h = divmod(hh, H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rl = oracle.forward(np64(t["q"][sl]), np64(t["k"][sl]), np64(t["v"][sl]), scale, causal=causal)
        check_fwd(o[sl], lse[sl], ro, rl, f"B{B} H{H} N{N} d{d} head {hh}")


BANDED = [
    # B, H, N, d, causal: heads whose K and V outgrow the forward's L2 budget,
    # so the persistent CTAs walk the items band by band (odd band counts,
    # ragged N, d = 64)
    (1, 12, 8192, 128, False),
    (2, 24, 16384, 64, True),
    (1, 24, 9000, 128, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", BANDED)
def test_forward_banded_item_order(fa, B, H, N, d, causal):
    """Every item of a banded launch is computed exactly where it belongs:
    outputs start as NaN and none is left; sampled whole heads against the
    oracle."""
    t = make_qkvdo(B, H, N, d, seed=90 + H, with_dout=False)
    scale = 1 / math.sqrt(d)
    q, k, v = (dev(t[n]) for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd(q, k, v, o, lse, scale, causal=causal)
    check_device_status(fa)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    o, lse = o.cpu(), lse.cpu()
    for hh in sorted(set([0, B * H - 1] + _sampled_heads(B * H, 2, seed=N))):
        b, h = divmod(hh, H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rl = oracle.forward(np64(t["q"][sl]), np64(t["k"][sl]), np64(t["v"][sl]), scale, causal=causal,
                                row_chunk=2048)
        check_fwd(o[sl], lse[sl], ro, rl, f"banded B{B} H{H} N{N} d{d} head {hh}")


def test_forward_workload_long_causal(fa):
    """N=16384 causal with x3 inputs: S would be 16 GiB.  Eight whole heads
    through the oracle (rows in chunks of 2048 full rows), and sampled rows of
    four more, including the first and last rows of the sequence."""
    w = WORKLOADS["fwd_b1h32n16384d128_causal_x3"]
    t = make_workload_inputs(w)
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]), causal=True, scale=w.scale)
    check_device_status(fa)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    o, lse = o.cpu(), lse.cpu()
    whole = _sampled_heads(w.H, 8, seed=3)
    for h in whole:
        sl = (slice(0, 1), slice(h, h + 1))
        q64, k64, v64 = np64(t["q"][sl]), np64(t["k"][sl]), np64(t["v"][sl])
        ro, rl = oracle.forward(q64, k64, v64, w.scale, causal=True, row_chunk=2048)
        pb = oracle.forward_error_bound(q64, k64, v64, w.scale, causal=True, row_chunk=2048)
        check_fwd(o[sl], lse[sl], ro, rl, f"N=16384 whole head {h}", pb)
    r = np.random.default_rng(3)
    rows = sorted(set([0, 1, 127, 128, w.N - 1] + r.choice(w.N, 59, replace=False).tolist()))
    for h in [x for x in range(w.H) if x not in whole][:4]:
        sl = (slice(0, 1), slice(h, h + 1))
        q64, k64, v64 = np64(t["q"][sl]), np64(t["k"][sl]), np64(t["v"][sl])
        ro, rl = oracle.forward_rows(q64, k64, v64, w.scale, 0, 0, rows, causal=True)
        pb = oracle.forward_error_bound(q64, k64, v64, w.scale, causal=True, rows=rows)[0, 0]
        check_fwd(o[0, h, rows], lse[0, h, rows], ro, rl, f"N=16384 head {h}", pb)


# --------------------------------------------------------------------------- #
# failure detection without a fault
# --------------------------------------------------------------------------- #
def test_bounded_wait_reports_timeout(fa):
    """A kernel waits on a barrier that nothing completes; the bounded wait gives
    up after 1 ms, the status word says FA_ERR_TIMEOUT, and the context stays
    usable for the next call."""
    assert fa.fa_debug_wait_timeout(1_000_000) == fa.FA_ERR_TIMEOUT
    assert fa.fa_get_device_error() == 0        # the read cleared it
    t = make_qkvdo(1, 1, 128, 64, seed=0, with_dout=False)
    o, lse = fa.forward(dev(t["q"]), dev(t["k"]), dev(t["v"]))
    check_device_status(fa)
    ro, rl = oracle.forward(np64(t["q"]), np64(t["k"]), np64(t["v"]), 1 / 8)
    check_fwd(o, lse, ro, rl, "after timeout")


# --------------------------------------------------------------------------- #
# backward
# --------------------------------------------------------------------------- #
def _run_fwd_bwd(fa, t, causal, scale, bm=None):
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    bmd = None if bm is None else dev(bm)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=bmd)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=bmd)
    check_device_status(fa)
    return dq, dk, dv


BWD_SMALL = [
    (1, 1, 128, 64, False, None),
    (1, 1, 128, 128, True, None),
    (2, 2, 256, 64, True, None),
    (1, 2, 384, 128, True, None),
    (1, 2, 384, 64, False, None),
    (2, 1, 512, 128, False, None),
    (1, 2, 512, 64, False, 0.3),
    (1, 2, 768, 128, False, 0.25),
]


@pytest.mark.parametrize("B,H,N,d,causal,p", BWD_SMALL)
def test_backward_small(fa, B, H, N, d, causal, p):
    t = make_qkvdo(B, H, N, d, seed=20 + N + d)
    scale = 1 / math.sqrt(d)
    bm = make_block_mask(N, seed=N + 1, p=p) if p is not None else None
    g = _run_fwd_bwd(fa, t, causal, scale, bm)
    f64 = {n: np64(t[n]) for n in ("q", "k", "v", "do")}
    ref, model = oracle_bwd(f64, scale, causal, None if bm is None else bm.numpy())
    check_bwd(g, ref, f"B{B} H{H} N{N} d{d} causal={causal} p={p}", model)


def test_backward_workload_n1024(fa):
    w = WORKLOADS["fwdbwd_b4h8n1024d64"]
    t = make_workload_inputs(w)
    g = _run_fwd_bwd(fa, t, w.causal, w.scale)
    f64 = {n: np64(t[n]) for n in ("q", "k", "v", "do")}
    ref, model = oracle_bwd(f64, w.scale)
    check_bwd(g, ref, w.name, model)


@pytest.mark.parametrize("name", ["fwdbwd_b2h16n4096d128_causal", "fwdbwd_b1h16n8192d128_blocksparse"])
def test_backward_workload_all_heads(fa, name):
    """Every head of the full-size workload through the oracle: per tensor
    and per tile relative L2, and every element inside the error model."""
    w = WORKLOADS[name]
    t = make_workload_inputs(w)
    bm = t.get("block_mask")
    g = _run_fwd_bwd(fa, t, w.causal, w.scale, bm)
    g = tuple(x.float().cpu() for x in g)
    for hh in range(w.B * w.H):
        b, h = divmod(hh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        f64 = {n: np64(t[n][sl]) for n in ("q", "k", "v", "do")}
        ref, model = oracle_bwd(f64, w.scale, w.causal, None if bm is None else bm.numpy())
        check_bwd(tuple(x[sl] for x in g), ref, f"{name} head {hh}", model)


def test_backward_fully_masked_blocks(fa):
    """A query block that sees nothing gets dQ = 0; a key block that no query
    sees gets dK = dV = 0."""
    B, H, N, d = 1, 2, 512, 128
    t = make_qkvdo(B, H, N, d, seed=78)
    bm = torch.ones(4, 4, dtype=torch.uint8)
    bm[1, :] = 0          # query block 1 sees nothing
    bm[:, 2] = 0          # key block 2 is seen by nobody
    g = _run_fwd_bwd(fa, t, False, 1 / math.sqrt(d), bm)
    f64 = {n: np64(t[n]) for n in ("q", "k", "v", "do")}
    ref, model = oracle_bwd(f64, 1 / math.sqrt(d), False, bm.numpy())
    check_bwd(g, ref, "fully masked blocks", model)
    dq, dk, dv = g
    assert torch.all(dq[:, :, 128:256] == 0)
    assert torch.all(dk[:, :, 256:384] == 0) and torch.all(dv[:, :, 256:384] == 0)


def test_backward_stages_match_fused_call(fa):
    """fa_bwd equals its three stages called one by one."""
    B, H, N, d = 1, 2, 512, 128
    t = make_qkvdo(B, H, N, d, seed=9)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    ws = fa.workspace(B, H, N, d, q.device)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_preprocess(o, do, lse, ws)
    fa.fa_bwd_main(q, k, v, do, None, dk2, dv2, ws, scale, fa.MASK_CAUSAL)
    fa.fa_bwd_dq_convert(ws, dq2, scale)
    check_device_status(fa)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    # dQ sums fp32 atomics in arrival order, so it is equal up to rounding only
    assert (dq.float() - dq2.float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item()


def test_backward_guard_bands(fa):
    B, H, N, d = 1, 1, 256, 64
    t = make_qkvdo(B, H, N, d, seed=11)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True)
    n, pad = B * H * N * d, 2048
    bufs = [torch.full((n + 2 * pad,), 5.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    outs = [b[pad:pad + n].view(B, H, N, d) for b in bufs]
    ws = fa.workspace(B, H, N, d, q.device)
    fa.fa_bwd(q, k, v, o, do, lse, *outs, ws, 1 / 8, causal=True)
    check_device_status(fa)
    for b in bufs:
        assert torch.all(b[:pad] == 5.0) and torch.all(b[pad + n:] == 5.0)


# --------------------------------------------------------------------------- #
# any sequence length: the last 128-row tile is partial
# --------------------------------------------------------------------------- #
RAGGED = [
    # B, H, N, d, mask
    (1, 1, 1, 64, "none"),
    (1, 2, 7, 128, "causal"),
    (2, 1, 100, 64, "causal"),
    (1, 2, 129, 128, "none"),
    (1, 1, 200, 64, "block"),
    (2, 2, 255, 128, "causal"),
    (1, 2, 333, 64, "none"),
    (1, 1, 450, 128, "block"),
    (1, 2, 700, 128, "causal"),
    (1, 1, 1001, 64, "causal"),
]


def _ragged_mask(N, seed):
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((nb, nb), generator=g) < 0.5).to(torch.uint8)
    bm.fill_diagonal_(1)
    return bm


@pytest.mark.parametrize("B,H,N,d,mask", RAGGED)
def test_ragged_sequence_length(fa, B, H, N, d, mask):
    t = make_qkvdo(B, H, N, d, seed=40 + N)
    scale = 1 / math.sqrt(d)
    causal = mask == "causal"
    bm = _ragged_mask(N, N) if mask == "block" else None
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    bmd = None if bm is None else dev(bm)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=bmd)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=bmd)
    check_device_status(fa)
    f64 = {n: np64(t[n]) for n in ("q", "k", "v", "do")}
    bmn = None if bm is None else bm.numpy()
    ro, rl = oracle.forward(f64["q"], f64["k"], f64["v"], scale, causal=causal, block_mask=bmn)
    check_fwd(o, lse, ro, rl, f"N={N} d={d} {mask}")
    ref, model = oracle_bwd(f64, scale, causal, bmn)
    check_bwd((dq, dk, dv), ref, f"N={N} d={d} {mask}", model)


ODD_TILE_MASKS = [
    # B, H, N, d, causal, mask seed: random block masks (p = 0.3) with rows of
    # unequal length, an odd number of query tiles (the last CTA has one),
    # the causal flag on top of a block mask, ragged N
    (1, 2, 1152, 128, False, 1152),
    (1, 2, 1408, 64, True, 1408),
    (2, 1, 1100, 128, False, 7),
]


@pytest.mark.parametrize("B,H,N,d,causal,seed", ODD_TILE_MASKS)
def test_block_mask_odd_tile_counts(fa, B, H, N, d, causal, seed):
    """Random block masks over an odd number of tiles, forward and backward:
    every element against the oracle."""
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((nb, nb), generator=g) < 0.3).to(torch.uint8)
    bm.fill_diagonal_(1)
    t = make_qkvdo(B, H, N, d, seed=60 + N)
    scale = 1 / math.sqrt(d)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    bmd = dev(bm)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=bmd)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=bmd)
    check_device_status(fa)
    f64 = {n: np64(t[n]) for n in ("q", "k", "v", "do")}
    ro, rl = oracle.forward(f64["q"], f64["k"], f64["v"], scale, causal=causal, block_mask=bm.numpy())
    check_fwd(o, lse, ro, rl, f"N={N} d={d} odd tiles")
    ref, model = oracle_bwd(f64, scale, causal, bm.numpy())
    check_bwd((dq, dk, dv), ref, f"N={N} d={d} odd tiles", model)


def _schedule_mask(nb, seed):
    """A block mask whose query-tile pairs (2t, 2t + 1) exercise the forward's
    round schedules: shared tiles at equal ranks at the start (then the
    tiles of one query tile alone), shared ranks with a gap, identical rows
    (every round shared), disjoint rows, an empty row beside a full one, one
    tile shared at different ranks; the remaining pairs random."""
    rows = [set(range(0, 5)) | {10, 11, 12}, set(range(0, 5)) | set(range(14, 20)),
            {1, 3, 5, 7, 9}, {0, 2, 4, 6, 8},
            set(range(10)), set(range(10)),
            set(), set(range(5, 10)),
            set(range(nb)), {nb - 1},
            {2, 5, 8, 11, 12, 13}, {2, 6, 8, 14, 15, 16}]
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((nb, nb), generator=g) < 0.3).to(torch.uint8)
    for qt, r in enumerate(rows):
        bm[qt] = 0
        for kt in r:
            bm[qt, kt] = 1
    return bm


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_round_schedules(fa, causal):
    """The block-mask forward runs each CTA's two query tiles in rounds whose
    schedule depends on which key tiles they share (shared first, or the r-th
    tile of each, with a shared load where those coincide); every schedule
    above against the oracle, every element, forward and backward."""
    B, H, N, d = 1, 2, 2560, 128
    nb = N // 128
    bm = _schedule_mask(nb, 123)
    t = make_qkvdo(B, H, N, d, seed=91)
    scale = 1 / math.sqrt(d)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=dev(bm))
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=dev(bm))
    check_device_status(fa)
    f64 = {n: np64(t[n]) for n in ("q", "k", "v", "do")}
    what = f"round schedules causal={causal}"
    ro, rl = oracle.forward(f64["q"], f64["k"], f64["v"], scale, causal=causal, block_mask=bm.numpy())
    check_fwd(o, lse, ro, rl, what)
    ref, model = oracle_bwd(f64, scale, causal, bm.numpy())
    check_bwd((dq, dk, dv), ref, what, model)


def test_ragged_outputs_stay_inside_their_rows(fa):
    """With N not a multiple of 128, nothing is written past row N - 1."""
    B, H, N, d = 1, 2, 200, 128
    t = make_qkvdo(B, H, N, d, seed=3)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    n, pad = B * H * N * d, 4096
    obuf = torch.full((n + pad,), 3.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * N + pad,), 3.0, dtype=torch.float32, device="cuda")
    o, lse = obuf[:n].view(B, H, N, d), lbuf[:B * H * N].view(B, H, N)
    fa.fa_fwd(q, k, v, o, lse, 1 / math.sqrt(d), causal=True)
    grads = [torch.full((n + pad,), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    ws = fa.workspace(B, H, N, d, q.device)
    fa.fa_bwd(q, k, v, o, do, lse, *(g[:n].view(B, H, N, d) for g in grads), ws, 1 / math.sqrt(d), causal=True)
    check_device_status(fa)
    assert torch.all(obuf[n:] == 3.0) and torch.all(lbuf[B * H * N:] == 3.0)
    for g in grads:
        assert torch.all(g[n:] == 3.0)


# --------------------------------------------------------------------------- #
# sliding-window and dilated block masks, and a block mask with the causal flag
# (masks from the library's host generators, checked against the oracle's own
# construction, then both paths run on them)
# --------------------------------------------------------------------------- #
PATTERNS = [
    # B, H, N, d, pattern, args, causal
    (1, 2, 1000, 64, "window", (2, 0), True),
    (1, 2, 2048, 128, "window", (3, 1), False),
    (1, 1, 1500, 128, "dilated", (2, 2), True),
    (2, 1, 1024, 64, "dilated", (3, 3), False),
    (1, 2, 777, 128, "window", (1, 0), True),
    (1, 1, 2560, 128, "random", 0.3, True),
    (1, 2, 1280, 64, "random", 0.5, True),
]


def _pattern_masks(fa, N, pattern, args):
    if pattern == "window":
        return fa.fa_block_mask_window(N, *args), oracle.window_block_mask(N, *args)
    if pattern == "dilated":
        return (fa.fa_block_mask_dilated(N, *args, causal=False),
                oracle.dilated_block_mask(N, *args, causal=False))
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(N)
    bm = (torch.rand((nb, nb), generator=g) < args).to(torch.uint8)
    bm.fill_diagonal_(1)
    return bm, bm.numpy()


@pytest.mark.parametrize("B,H,N,d,pattern,args,causal", PATTERNS)
def test_window_dilated_and_causal_block_masks(fa, B, H, N, d, pattern, args, causal):
    bm, bm_ref = _pattern_masks(fa, N, pattern, args)
    np.testing.assert_array_equal(bm.numpy(), bm_ref)
    t = make_qkvdo(B, H, N, d, seed=60 + N)
    scale = 1 / math.sqrt(d)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=dev(bm))
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=dev(bm))
    check_device_status(fa)
    f64 = {n: np64(t[n]) for n in ("q", "k", "v", "do")}
    what = f"N={N} d={d} {pattern}{args} causal={causal}"
    ro, rl = oracle.forward(f64["q"], f64["k"], f64["v"], scale, causal=causal, block_mask=bm_ref)
    check_fwd(o, lse, ro, rl, what)
    ref, model = oracle_bwd(f64, scale, causal, bm_ref)
    check_bwd((dq, dk, dv), ref, what, model)


def test_causal_window_long_sequence_sampled_rows(fa):
    """Causal sliding window (16 blocks back) at N = 16384, d = 128: sampled
    query rows of two heads through the oracle, forward and backward dQ."""
    B, H, N, d = 1, 2, 16384, 128
    t = make_qkvdo(B, H, N, d, seed=77)
    scale = 1 / math.sqrt(d)
    bm = fa.fa_block_mask_window(N, 16, 0)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=scale, block_mask=dev(bm))
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, block_mask=dev(bm))
    check_device_status(fa)
    bm_ref = oracle.window_block_mask(N, 16, 0)
    rows = np.array([0, 1, 127, 128, 2047, 2048, 5000, 9999, 16256, 16383])
    for h in range(H):
        f64 = {n: np64(t[n][:, h:h + 1]) for n in ("q", "k", "v", "do")}
        ro, rl = oracle.forward_rows(f64["q"], f64["k"], f64["v"], scale, 0, 0, rows, causal=True, block_mask=bm_ref)
        check_fwd(o[0, h, rows], lse[0, h, rows], ro, rl, f"causal window N=16384 head {h}")
        rdq = oracle.backward_rows_dq(f64["q"], f64["k"], f64["v"], f64["do"], scale, 0, 0, rows,
                                      causal=True, block_mask=bm_ref)
        err = rel_l2(dq[0, h, rows], rdq)
        assert err <= GRAD_RTOL, f"h={h} dQ rows rel-L2 {err}"


# --------------------------------------------------------------------------- #
# the largest size the ABI accepts: B*H*N*d just under 2^31 elements, where
# any 32-bit offset would overflow (inputs drawn on the device from a seeded
# generator; sampled rows of two heads through the oracle)
# --------------------------------------------------------------------------- #
def test_forward_backward_at_the_index_limit(fa):
    B, H, N, d = 1, 127, 131072, 128
    assert B * H * N * d < 2 ** 31 and B * (H + 1) * N * d >= 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(2024)
    q, k, v, do = (torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    check_device_status(fa)
    tail = np.arange(N - 256, N)
    for h in (0, H - 1):
        f64 = {n: x[:, h:h + 1].double().cpu().numpy() for n, x in (("q", q), ("k", k), ("v", v), ("do", do))}
        rows = np.array([0, 1, 127, 128, 65535, 65536, N - 129, N - 1])
        ro, rl = oracle.forward_rows(f64["q"], f64["k"], f64["v"], scale, 0, 0, rows, causal=True)
        check_fwd(o[0, h, rows], lse[0, h, rows], ro, rl, f"index limit head {h}")
        rdq = oracle.backward_rows_dq(f64["q"], f64["k"], f64["v"], f64["do"], scale, 0, 0, rows, causal=True)
        assert rel_l2(dq[0, h, rows], rdq) <= GRAD_RTOL, f"index limit head {h}: dQ rows"
        # keys N-256.. are seen only by query rows N-256.. (causal): their
        # dK and dV are exactly the contributions of those rows
        _, dkp, dvp, _, _ = oracle.backward_rows(f64["q"], f64["k"], f64["v"], f64["do"], scale, 0, 0, tail,
                                                 causal=True)
        assert rel_l2(dk[0, h, tail], dkp[tail]) <= GRAD_RTOL, f"index limit head {h}: dK tail"
        assert rel_l2(dv[0, h, tail], dvp[tail]) <= GRAD_RTOL, f"index limit head {h}: dV tail"
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- #
# many short heads: large grids of one-tile problems
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_many_short_heads(fa, d, causal):
    B, H, N = 32, 32, 128
    t = make_qkvdo(B, H, N, d, seed=500 + d)
    scale = 1 / math.sqrt(d)
    q, k, v, do = (dev(t[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    check_device_status(fa)
    for b, h in ((0, 0), (13, 7), (31, 31)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        f64 = {n: np64(t[n][sl]) for n in ("q", "k", "v", "do")}
        ro, rl = oracle.forward(f64["q"], f64["k"], f64["v"], scale, causal=causal)
        check_fwd(o[sl], lse[sl], ro, rl, f"B32 H32 N128 d{d} head ({b}, {h})")
        ref, model = oracle_bwd(f64, scale, causal)
        check_bwd((dq[sl], dk[sl], dv[sl]), ref, f"B32 H32 N128 d{d} head ({b}, {h})", model)
