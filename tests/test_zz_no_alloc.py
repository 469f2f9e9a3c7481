"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

A serving process whose memory pool reserved the whole device at start-up, or
a plugin whose host framework owns the allocator, cannot cudaMalloc the fp32
dQ accumulator that fa_bwd needs as its workspace.  fa_bwd_noalloc runs the
same backward with that workspace in a static device array inside libfa.so.

The GPU test compares it with fa_bwd (caller-allocated workspace) on two calls
in a row on different problems: the array keeps the previous call's
contents, so the second call also shows that each call starts from a cleared
accumulator.  This file is named to be collected last.
"""
import ctypes
import math

import pytest
import torch

from attn_fwd_gb300.inputs import make_qkvdo

GRAD_RTOL = 2e-2   # the relative L2 bound the parity tests use for dQ, dK, dV


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


def test_noalloc_rejects_problems_beyond_its_scratch(fa):
    """Checked on the host before any device work: no GPU needed."""
    P = ctypes.c_void_p(4096)
    # B*H*N*d = 2^27 elements: a 512 MiB fp32 accumulator, beyond 64 MiB
    rc = fa.load().fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, 1, 64, 16384, 128, 0.088, 1, ctypes.c_void_p(0))
    assert rc == fa.FA_ERR_SCRATCH
    assert "static scratch" in fa.status_string(rc)
    limit = 64 << 20
    assert fa.fa_bwd_workspace_bytes(2, 16, 4096, 128) > limit     # the N=4096 workload needs fa_bwd
    assert fa.fa_bwd_workspace_bytes(2, 4, 1024, 128) <= limit


def _rel_l2(a, b):
    a, b = a.float(), b.float()
    return ((a - b).norm() / b.norm().clamp_min(1e-30)).item()


def _problem(B, H, N, d, causal, seed):
    t = make_qkvdo(B, H, N, d, seed=seed)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    return dict(q=q, k=k, v=v, do=do, causal=causal, scale=1 / math.sqrt(d))


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(fa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    problems = [_problem(2, 4, 1024, 128, True, 31), _problem(1, 3, 768, 64, False, 32)]
    for pr in problems:
        q, k, v, do = pr["q"], pr["k"], pr["v"], pr["do"]
        o, lse = fa.forward(q, k, v, causal=pr["causal"], scale=pr["scale"])
        ref = fa.backward(q, k, v, o, lse, do, causal=pr["causal"], scale=pr["scale"])
        pr.update(o=o, lse=lse, ref=ref)
    torch.cuda.synchronize()
    # two calls in a row through the C ABI, on different problems
    for pr in problems:
        dq, dk, dv = (torch.full_like(pr["q"], float("nan")) for _ in range(3))
        fa.fa_bwd_noalloc(pr["q"], pr["k"], pr["v"], pr["o"], pr["do"], pr["lse"], dq, dk, dv, pr["scale"],
                          causal=pr["causal"])
        torch.cuda.synchronize()
        assert fa.fa_get_device_error() == 0
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), pr["ref"]):
            assert torch.isfinite(got).all(), name
            err = _rel_l2(got, want)
            assert err <= GRAD_RTOL, f"{name} differs from fa_bwd: rel-L2 {err}"
