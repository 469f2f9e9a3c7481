"""The library used from several host threads at once, each on its own
stream: the tensor-map cache, the per-device state and the host-streamed
entry point's lock are shared.  Every thread's results must equal the ones
a single thread gets on the same inputs (O, LSE, dK, dV bit for bit; dQ,
summed with fp32 atomics in a run-dependent order, to within one bf16
rounding step)."""
import math
import threading

import pytest
import torch

from attn_fwd_gb300.inputs import make_decode_inputs, make_qkvdo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import attn_fwd_gb300.fa as fa
    fa.load()
    return fa


def _same(name, a, b):
    if name == "dq":
        torch.testing.assert_close(a.float(), b.float(), rtol=2 ** -7, atol=1e-4)
    else:
        assert torch.equal(a, b), name


def _run_threads(work, n):
    errors = []

    def body(i):
        try:
            work(i)
        except BaseException as e:          # reported by the main thread
            errors.append(e)

    ts = [threading.Thread(target=body, args=(i,)) for i in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errors:
        raise errors[0]


def test_forward_backward_from_two_threads(fa):
    shapes = [(2, 4, 1024, 128, True), (1, 6, 777, 64, False)]
    inputs = [make_qkvdo(B, H, N, d, seed=100 + i) for i, (B, H, N, d, _) in enumerate(shapes)]

    def step(i, stream):
        B, H, N, d, causal = shapes[i]
        with torch.cuda.stream(stream):
            t = {n: inputs[i][n].cuda(non_blocking=False) for n in ("q", "k", "v", "do")}
            o, lse = fa.forward(t["q"], t["k"], t["v"], causal=causal, stream=stream)
            dq, dk, dv = fa.backward(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, stream=stream)
        stream.synchronize()
        return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}

    ref = [step(i, torch.cuda.Stream()) for i in range(len(shapes))]
    got = [[None] * 10 for _ in shapes]

    def work(i):
        s = torch.cuda.Stream()
        for r in range(10):
            got[i][r] = step(i, s)

    _run_threads(work, len(shapes))
    assert fa.fa_get_device_error() == 0
    for i in range(len(shapes)):
        for r in range(10):
            for name in ref[i]:
                _same(name, got[i][r][name], ref[i][name])


def test_decode_and_host_streamed_steps_from_two_threads(fa):
    """One thread decodes, the other runs the host-streamed forward and
    backward (its library-owned streams) on the same device."""
    dec = make_decode_inputs(2, 8, 4, 5000, 128, seed=9)
    qkv = make_qkvdo(1, 20, 2048, 128, seed=10)
    host = {n: qkv[n].pin_memory() for n in ("q", "k", "v", "do")}
    ws = torch.empty(fa.fa_fwd_bwd_host_workspace_bytes(1, 20, 2048, 128), dtype=torch.uint8, device="cuda")
    dq_, dk_, dv_ = (dec[n].cuda() for n in ("q", "k", "v"))
    torch.cuda.synchronize()

    def decode(stream):
        with torch.cuda.stream(stream):
            o, lse = fa.decode(dq_, dk_, dv_, causal=True, stream=stream)
        stream.synchronize()
        return {"o": o, "lse": lse}

    def streamed():
        r = fa.forward_backward_host(host["q"], host["k"], host["v"], host["do"], causal=True, ws=ws)
        torch.cuda.synchronize()
        return dict(zip(("o", "lse", "dq", "dk", "dv"), r))

    ref_dec, ref_host = decode(torch.cuda.Stream()), streamed()
    out = {"dec": [], "host": []}

    def work(i):
        if i == 0:
            s = torch.cuda.Stream()
            for _ in range(10):
                out["dec"].append(decode(s))
        else:
            for _ in range(3):
                out["host"].append(streamed())

    _run_threads(work, 2)
    assert fa.fa_get_device_error() == 0
    for r in out["dec"]:
        for name in ref_dec:
            _same(name, r[name], ref_dec[name])
    for r in out["host"]:
        for name in ref_host:
            _same(name, r[name], ref_host[name])
