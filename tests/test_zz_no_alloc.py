"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

A serving process whose memory pool reserved the whole device at start-up, or
a plugin whose host framework owns the allocator, cannot cudaMalloc the fp32
dQ accumulator that fa_bwd needs as its workspace.  fa_bwd_noalloc runs the
same backward with that workspace in a static device array inside libfa.so.

The GPU test calls it through the C ABI on several problems in a row (the
array keeps the previous call's contents, so each later call also shows that
a call starts from a cleared accumulator): a causal d = 128 problem, a d = 64
one, a ragged N = 1000 (padded -D/-LSE rows inside the array) and one whose
workspace ends just under the array's end.  Each is compared with fa_bwd on a
caller-allocated workspace, which runs the same kernels: dK and dV bit for
bit, dQ up to the order of its fp32 atomic additions.  The ragged problem is
also compared with the fp64 oracle directly, and the device's free memory is
read around a call to show that it allocates nothing.  This file is named to
be collected last.
"""
import ctypes
import math

import pytest
import torch

from attn_fwd_gb300.inputs import make_qkvdo
from tests.parity_checks import check_bwd, oracle_bwd

LIMIT = 64 << 20      # FA_NOALLOC_SCRATCH_BYTES


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
    assert fa.fa_bwd_workspace_bytes(2, 16, 4096, 128) > LIMIT     # the N=4096 workload needs fa_bwd
    assert fa.fa_bwd_workspace_bytes(2, 4, 1024, 128) <= LIMIT
    # the largest problem below uses the array up to within 2 MiB of its end
    assert LIMIT - (2 << 20) < fa.fa_bwd_workspace_bytes(1, 31, 4096, 128) <= LIMIT
    assert fa.fa_bwd_workspace_bytes(1, 32, 4096, 128) > LIMIT


def _problem(B, H, N, d, causal, seed):
    t = make_qkvdo(B, H, N, d, seed=seed)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    return dict(t=t, q=q, k=k, v=v, do=do, causal=causal, scale=1 / math.sqrt(d), what=f"B{B} H{H} N{N} d{d}")


def _rel_l2(a, b):
    a, b = a.float(), b.float()
    return ((a - b).norm() / b.norm().clamp_min(1e-30)).item()


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_on_calls_in_a_row(fa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    problems = [_problem(2, 4, 1024, 128, True, 31), _problem(1, 3, 768, 64, False, 32),
                _problem(1, 2, 1000, 128, True, 33), _problem(1, 31, 4096, 128, True, 34)]
    for pr in problems:
        q, k, v, do = pr["q"], pr["k"], pr["v"], pr["do"]
        o, lse = fa.forward(q, k, v, causal=pr["causal"], scale=pr["scale"])
        ref = fa.backward(q, k, v, o, lse, do, causal=pr["causal"], scale=pr["scale"])
        pr.update(o=o, lse=lse, ref=ref)
    torch.cuda.synchronize()
    # calls in a row through the C ABI, on different problems; the last one
    # twice, with the device's free memory read around the second call
    for n, pr in enumerate(problems + problems[-1:]):
        dq, dk, dv = (torch.full_like(pr["q"], float("nan")) for _ in range(3))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        fa.fa_bwd_noalloc(pr["q"], pr["k"], pr["v"], pr["o"], pr["do"], pr["lse"], dq, dk, dv, pr["scale"],
                          causal=pr["causal"])
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert fa.fa_get_device_error() == 0
        if n == len(problems):
            assert free_after >= free_before, f"device memory dropped by {free_before - free_after} bytes"
        rq, rk, rv = pr["ref"]
        assert torch.equal(dk, rk), f"{pr['what']}: dK differs from fa_bwd"
        assert torch.equal(dv, rv), f"{pr['what']}: dV differs from fa_bwd"
        assert torch.isfinite(dq).all(), pr["what"]
        err = _rel_l2(dq, rq)
        assert err <= 1e-4, f"{pr['what']}: dQ differs from fa_bwd by rel-L2 {err}"
        one_ulp = ((dq.float() - rq.float()).abs() <= 2.0 ** -7 * rq.float().abs() + 1e-6 * rq.float().abs().max())
        assert one_ulp.all(), f"{pr['what']}: dQ differs from fa_bwd by more than one bf16 step"
        if pr["what"] == "B1 H2 N1000 d128":
            f64 = {x: pr["t"][x].double().numpy() for x in ("q", "k", "v", "do")}
            ref, model = oracle_bwd(f64, pr["scale"], pr["causal"])
            check_bwd((dq, dk, dv), ref, f"fa_bwd_noalloc {pr['what']} vs the oracle", model)
