"""The debug build, libfa_debug.so: the same sources compiled with FA_DEBUG,
whose kernels check their computed indices against the extent of the buffer
they access (the block mask, the -LSE/-D rows the backward copies, the dQ
accumulator, the output rows) and, on a failed check, record FA_ERR_BOUNDS in
the status word and skip the access instead of faulting.  It stands in for
the memory checker, which is not available on the GPUs these tests run on.

CPU: it builds and exports the same entry points as libfa.so.  GPU: on
ragged, causal and block-masked problems no check fires and the outputs are
those of the release build (O, LSE, dK, dV bit for bit; dQ, summed by fp32
atomics in arrival order, within one bf16 step).
"""
import ctypes
import math
import subprocess

import pytest
import torch

from attn_fwd_gb300 import build as fa_build
from attn_fwd_gb300.inputs import make_qkvdo


@pytest.fixture(scope="module")
def debug_lib():
    path = fa_build.build(debug=True)
    return ctypes.CDLL(path)


def _exports(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if " T " in line and line.split()[-1].startswith("fa_")}


def test_debug_build_exports_the_same_entry_points(debug_lib):
    release = fa_build.build()
    assert _exports(fa_build.LIB_DEBUG) == _exports(release)
    debug_lib.fa_status_string.restype = ctypes.c_char_p
    assert b"FA_ERR_BOUNDS" in debug_lib.fa_status_string(-8)


CASES = [
    # B, H, N, d, mask
    (1, 2, 1000, 128, "causal"),
    (1, 2, 700, 64, "block"),
    (2, 2, 384, 64, "none"),
    (1, 1, 1300, 128, "block_causal"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,mask", CASES)
def test_debug_build_checks_pass_and_match_release(debug_lib, B, H, N, d, mask):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attn_fwd_gb300.fa as fa
    fa.load()
    t = make_qkvdo(B, H, N, d, seed=300 + N)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1 / math.sqrt(d)
    causal = mask in ("causal", "block_causal")
    bm = None
    if mask.startswith("block"):
        nb = (N + 127) // 128
        g = torch.Generator().manual_seed(N)
        bm = (torch.rand((nb, nb), generator=g) < 0.4).to(torch.uint8)
        bm.fill_diagonal_(1)
        bm = bm.cuda()
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, block_mask=bm)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, block_mask=bm)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    # the same calls through the debug library
    L = debug_lib
    vp = ctypes.c_void_p
    st = vp(torch.cuda.current_stream().cuda_stream)
    ptr = lambda x: vp(x.data_ptr())
    o2, dq2, dk2, dv2 = (torch.full_like(q, float("nan")) for _ in range(4))
    lse2 = torch.full_like(lse, float("nan"))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    L.fa_fwd_blocksparse.argtypes = [vp] * 6 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, vp]
    L.fa_fwd.argtypes = [vp] * 5 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, vp]
    L.fa_bwd.argtypes = [vp] * 10 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, vp]
    L.fa_bwd_blocksparse.argtypes = [vp] * 11 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, vp]
    L.fa_get_device_error.argtypes = [vp]
    c = int(causal)
    if bm is None:
        rc = L.fa_fwd(ptr(q), ptr(k), ptr(v), ptr(o2), ptr(lse2), B, H, N, d, scale, c, st)
        assert rc == 0
        rc = L.fa_bwd(ptr(q), ptr(k), ptr(v), ptr(o2), ptr(do), ptr(lse2), ptr(dq2), ptr(dk2), ptr(dv2), ptr(ws),
                      B, H, N, d, scale, c, st)
    else:
        rc = L.fa_fwd_blocksparse(ptr(q), ptr(k), ptr(v), ptr(o2), ptr(lse2), ptr(bm), B, H, N, d, scale, c, st)
        assert rc == 0
        rc = L.fa_bwd_blocksparse(ptr(q), ptr(k), ptr(v), ptr(o2), ptr(do), ptr(lse2), ptr(bm), ptr(dq2), ptr(dk2),
                                  ptr(dv2), ptr(ws), B, H, N, d, scale, c, st)
    assert rc == 0
    assert L.fa_get_device_error(st) == 0, "a device index check fired"
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    diff = (dq.float() - dq2.float()).abs()
    assert bool((diff <= 2.0 ** -7 * dq.float().abs() + 1e-6 * dq.float().abs().max()).all())
