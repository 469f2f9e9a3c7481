"""Stream capture.  The device-resident entry points (fa_fwd*, fa_bwd*,
fa_decode) enqueue kernel launches on the caller's stream and nothing else:
no allocation, no copy, no synchronisation.  So a forward + backward step, or
a decoding step, can be captured into a CUDA graph once and replayed with new
values copied into the captured buffers.  Each replay must reproduce an eager
call on the same values: O, LSE, dK, dV and decode outputs bit for bit (their
schedules are fixed), dQ up to the order of its fp32 reductions.

The first call of an entry point on a device sets up per-device state (the
architecture check, the status word's address, the kernels' shared-memory
limits), so every test calls eagerly once before capturing.
"""
import math

import numpy as np
import pytest
import torch

from attn_fwd_gb300.inputs import make_block_mask, make_decode_inputs, make_qkvdo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


def _status_ok(fa):
    torch.cuda.synchronize()
    rc = fa.fa_get_device_error()
    assert rc == 0, fa.status_string(rc)


def _capture(fn):
    """Warm up on a side stream, then capture fn into a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


STEPS = [
    # B, H, N, d, mode
    (2, 4, 1024, 128, "causal"),
    (1, 4, 2048, 64, "none"),
    (1, 2, 2048, 128, "block"),
    (1, 2, 1000, 128, "dropout"),
]


@pytest.mark.parametrize("B,H,N,d,mode", STEPS)
def test_forward_backward_graph_replay(fa, B, H, N, d, mode):
    causal = mode in ("causal", "dropout")
    scale = 1 / math.sqrt(d)
    t0 = make_qkvdo(B, H, N, d, seed=300 + N)
    q, k, v, do = (t0[n].cuda() for n in ("q", "k", "v", "do"))
    bm = make_block_mask(N, seed=5, p=0.3).cuda() if mode == "block" else None
    drop_p, drop_seed = (0.15, 77) if mode == "dropout" else (0.0, 0)
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws = fa.workspace(B, H, N, d, q.device)

    def step():
        if mode == "dropout":
            fa.fa_fwd_dropout(q, k, v, o, lse, None, scale, causal, drop_p, drop_seed)
            fa.fa_bwd_dropout(q, k, v, o, do, lse, None, dq, dk, dv, ws, scale, causal, drop_p, drop_seed)
        elif bm is not None:
            fa.fa_fwd_blocksparse(q, k, v, o, lse, bm, scale, causal)
            fa.fa_bwd_blocksparse(q, k, v, o, do, lse, bm, dq, dk, dv, ws, scale, causal)
        else:
            fa.fa_fwd(q, k, v, o, lse, scale, causal)
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal)

    g = _capture(step)
    for seed in (301, 302):
        t = make_qkvdo(B, H, N, d, seed=seed)
        for name, dst in (("q", q), ("k", k), ("v", v), ("do", do)):
            dst.copy_(t[name])
        g.replay()
        _status_ok(fa)
        ro, rl = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=bm, dropout_p=drop_p, seed=drop_seed)
        rdq, rdk, rdv = fa.backward(q, k, v, ro, rl, do, causal=causal, scale=scale, block_mask=bm,
                                    dropout_p=drop_p, seed=drop_seed)
        _status_ok(fa)
        assert torch.equal(o, ro) and torch.equal(lse, rl), f"{mode}: forward replay differs from eager"
        assert torch.equal(dk, rdk) and torch.equal(dv, rdv), f"{mode}: dK/dV replay differs from eager"
        a, b = dq.float(), rdq.float()
        rel = (torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b)).item()
        assert rel <= 1e-3, f"{mode}: dQ replay vs eager rel-L2 {rel}"


def test_decode_graph_replay(fa):
    B, H, Nq, Nk, d = 4, 8, 2, 5000, 128
    scale = 1 / math.sqrt(d)
    t0 = make_decode_inputs(B, H, Nq, Nk, d, seed=310)
    q, k, v = (t0[n].cuda() for n in ("q", "k", "v"))
    seqlens = torch.tensor([Nk, 4000, 17, 2500], dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    n = fa.fa_decode_workspace_bytes(B, H, Nq, Nk, d)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")

    def step():
        fa.fa_decode(q, k, v, o, lse, seqlens, scale, True, ws if n else None)

    g = _capture(step)
    for seed, lens in ((311, [3000, Nk, 1, 4096]), (312, [128, 129, Nk - 1, 64])):
        t = make_decode_inputs(B, H, Nq, Nk, d, seed=seed)
        for name, dst in (("q", q), ("k", k), ("v", v)):
            dst.copy_(t[name])
        seqlens.copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        _status_ok(fa)
        ro, rl = fa.decode(q, k, v, seqlens_k=seqlens, causal=True, scale=scale)
        _status_ok(fa)
        assert torch.equal(o, ro) and torch.equal(lse, rl), "decode replay differs from eager"
        assert np.isfinite(o.float().cpu().numpy()).all()
