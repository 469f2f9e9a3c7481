"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from attn_fwd_gb300 import build
    import attn_fwd_gb300.fa as fa
    build.build()
    return fa.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    return sorted(set(re.findall(r"FA_API\s+[^;(]*?\b(fa_\w+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared()
    for must in ("fa_fwd", "fa_bwd", "fa_fwd_blocksparse", "fa_bwd_blocksparse",
                 "fa_bwd_workspace_bytes", "fa_get_device_error", "fa_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    # and nothing else of ours leaks out of the shared object
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = sorted(set(re.findall(r"\bT (fa_\w+)", out)))
    assert exported == _declared()


def test_python_binding_covers_every_entry_point(lib):
    import attn_fwd_gb300.fa as fa
    for name in _declared():
        assert callable(getattr(fa, name)), name


def test_status_strings(lib):
    import attn_fwd_gb300.fa as fa
    for code in range(0, -7, -1):
        assert fa.status_string(code).startswith("FA_")
    assert fa.status_string(12345) == "unknown fa_status"
    assert fa.fa_version() >= 100


def test_workspace_bytes(lib):
    import attn_fwd_gb300.fa as fa
    B, H, N, d = 2, 16, 4096, 128
    n = fa.fa_bwd_workspace_bytes(B, H, N, d)
    assert n == B * H * N * d * 4 + 2 * B * H * N * 4
    assert n % 256 == 0
    # -D and -LSE rows are padded to a multiple of 128 per head
    assert fa.fa_bwd_workspace_bytes(1, 3, 200, 64) == 1 * 3 * 200 * 64 * 4 + 2 * 3072
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 64) == 256 + 2 * 512
    assert fa.fa_bwd_workspace_bytes(0, 1, 128, 64) == 0
    assert fa.fa_bwd_workspace_bytes(1 << 20, 1 << 10, 128, 128) == 0   # 2^31 elements or more


P = ctypes.c_void_p(4096)   # 16-byte aligned dummy pointers; never dereferenced on these paths
NULL = ctypes.c_void_p(0)
ODD = ctypes.c_void_p(4096 + 8)


@pytest.mark.parametrize("args,expect", [
    ((NULL, P, P, P, P, 1, 1, 128, 64, 0.125, 0), -1),          # null q
    ((P, P, P, P, ODD, 1, 1, 128, 64, 0.125, 0), -1),           # misaligned lse
    ((P, P, P, P, P, 0, 1, 128, 64, 0.125, 0), -1),             # B = 0
    ((P, P, P, P, P, 1, 1, 128, 96, 0.125, 0), -2),             # d not built
    ((P, P, P, P, P, 1, 1, 128, 64, float("nan"), 0), -1),      # scale not finite
    ((P, P, P, P, P, 1, 1, 128, 64, -1.0, 0), -1),              # scale <= 0
    ((P, P, P, P, P, 65536, 256, 1024, 128, 0.1, 0), -1),       # 2^31 elements or more
])
def test_fwd_rejects_bad_arguments(lib, args, expect):
    assert lib.fa_fwd(*args, NULL) == expect


def test_blocksparse_requires_mask(lib):
    assert lib.fa_fwd_blocksparse(P, P, P, P, P, NULL, 1, 1, 128, 64, 0.125, 0, NULL) == -1
    assert lib.fa_fwd_blocksparse(P, P, P, P, P, NULL, 1, 1, 128, 64, 0.125, 1, NULL) == -1
    assert lib.fa_bwd_blocksparse(P, P, P, P, P, P, NULL, P, P, P, P, 1, 1, 128, 64, 0.125, 0, NULL) == -1
    assert lib.fa_bwd_main(P, P, P, P, NULL, P, P, P, 1, 1, 128, 64, 0.125, 3, 0.0, 0, NULL) == -1


def test_bwd_rejects_bad_arguments(lib):
    ws = ctypes.c_void_p(4096 + 16)       # 16- but not 256-byte aligned
    assert lib.fa_bwd(P, P, P, P, P, P, P, P, P, NULL, 1, 1, 128, 64, 0.125, 0, NULL) == -1
    assert lib.fa_bwd_main(P, P, P, P, NULL, P, P, ws, 1, 1, 128, 64, 0.125, 0, 0.0, 0, NULL) == -1
    assert lib.fa_bwd_main(P, P, P, P, NULL, P, P, P, 1, 1, 128, 64, 0.125, 7, 0.0, 0, NULL) == -1
    assert lib.fa_bwd_main(P, P, P, P, NULL, P, P, P, 1, 1, 128, 64, 0.125, 4, 0.0, 0, NULL) == -1
    assert lib.fa_bwd_main(P, P, P, P, NULL, P, P, P, 1, 1, 128, 64, 0.125, 2, 0.0, 0, NULL) == -1
    assert lib.fa_bwd_preprocess(P, P, P, P, 1, 1, 100, 96, NULL) == -2
    assert lib.fa_bwd_preprocess(P, P, NULL, P, 1, 1, 100, 64, NULL) == -1    # lse required here
    # block masks are limited to 1024 tiles per row
    assert lib.fa_fwd_blocksparse(P, P, P, P, P, P, 1, 1, 1024 * 128 + 1, 64, 0.125, 0, NULL) == -2
    assert lib.fa_bwd_dq_convert(P, P, 1, 1, 128, 64, 0.0, NULL) == -1


def test_host_streamed_entry_checks(lib):
    """fa_fwd_bwd_host: workspace sizing and argument checks on the host."""
    import attn_fwd_gb300.fa as fa
    # two buffer sets of G heads: 8 bf16 tensors, LSE and the backward workspace
    # each; G covers two backward waves (2 * 152 / key tiles), at most 8
    # chunks, heads spread evenly: 4 chunks of 8 here
    B, H, N, d = 2, 16, 4096, 128
    G = 8
    per_set = 8 * G * N * d * 2 + G * N * 4 + fa.fa_bwd_workspace_bytes(1, G, N, d)
    assert fa.fa_fwd_bwd_host_workspace_bytes(B, H, N, d) == 2 * per_set
    assert fa.fa_fwd_bwd_host_workspace_bytes(1, 1, 128, 64) == 2 * (8 * 128 * 64 * 2 + 512 +
                                                                      fa.fa_bwd_workspace_bytes(1, 1, 128, 64))
    assert fa.fa_fwd_bwd_host_workspace_bytes(0, 1, 128, 64) == 0
    assert fa.fa_fwd_bwd_host_workspace_bytes(1, 1, 128, 96) == 0
    ws = ctypes.c_void_p(4096)
    big = 1 << 40
    args = [P] * 9 + [NULL, ws, big, 1, 1, 128, 64, 0.125, 1, NULL]
    for i in range(9):                                  # each host buffer is required
        a = list(args)
        a[i] = NULL
        assert lib.fa_fwd_bwd_host(*a) == -1
    a = list(args); a[10] = NULL
    assert lib.fa_fwd_bwd_host(*a) == -1                # no workspace
    a = list(args); a[10] = ctypes.c_void_p(4096 + 16)
    assert lib.fa_fwd_bwd_host(*a) == -1                # workspace not 256-byte aligned
    a = list(args); a[11] = 1024
    assert lib.fa_fwd_bwd_host(*a) == -1                # workspace too small
    a = list(args); a[15] = 96
    assert lib.fa_fwd_bwd_host(*a) == -2                # head dim not built
    a = list(args); a[16] = 0.0
    assert lib.fa_fwd_bwd_host(*a) == -1                # scale


def test_host_streamed_forward_checks(lib):
    """fa_fwd_host: workspace sizing (two sets of q, k, v, O and LSE for G
    heads, G covering two forward waves of 152 CTAs) and argument checks."""
    import attn_fwd_gb300.fa as fa
    B, H, N, d = 1, 32, 16384, 128
    G = 5                                    # one CTA per query-tile pair: 64 per head -> 5 heads
    assert fa.fa_fwd_host_workspace_bytes(B, H, N, d) == 2 * (4 * G * N * d * 2 + G * N * 4)
    assert fa.fa_fwd_host_workspace_bytes(0, 1, 128, 64) == 0
    ws = ctypes.c_void_p(4096)
    args = [P, P, P, P, P, NULL, ws, 1 << 40, 1, 1, 128, 64, 0.125, 1, NULL]
    for i in range(5):                       # q, k, v, o, lse are required
        a = list(args)
        a[i] = NULL
        assert lib.fa_fwd_host(*a) == -1
    a = list(args); a[6] = ctypes.c_void_p(4096 + 16)
    assert lib.fa_fwd_host(*a) == -1         # workspace not 256-byte aligned
    a = list(args); a[7] = 1024
    assert lib.fa_fwd_host(*a) == -1         # workspace too small
    a = list(args); a[11] = 96
    assert lib.fa_fwd_host(*a) == -2         # head dim not built


def test_timeout_setter(lib):
    assert lib.fa_set_wait_timeout_ns(0) == -1
    assert lib.fa_set_wait_timeout_ns(2_000_000_000) == 0
    assert lib.fa_debug_wait_timeout(0, NULL) == -1
    assert lib.fa_debug_wait_timeout(5_000_000_000, NULL) == -1


def test_valid_call_without_gpu_fails_loudly(lib):
    """With no usable CUDA device a valid call reports an error code; it never
    computes anything on the host."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = lib.fa_fwd(P, P, P, P, P, 1, 1, 128, 64, 0.125, 0, NULL)
    assert rc in (-6, -3)


# --------------------------------------------------------------------------- #
# block-mask generators (host functions: no GPU needed), against the oracle's
# own construction from the definitions
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("N,left,right", [
    (1, 0, 0), (128, 3, 0), (300, 1, 1), (1000, 2, 0), (1024, 0, 3), (4096, 5, 2),
    (8192, 64, 64), (131072, 16, 0),
])
def test_window_mask_matches_oracle(lib, N, left, right):
    import numpy as np
    import attn_fwd_gb300.fa as fa
    import oracle
    got = fa.fa_block_mask_window(N, left, right).numpy()
    np.testing.assert_array_equal(got, oracle.window_block_mask(N, left, right))


@pytest.mark.parametrize("N,window,dilation,causal", [
    (1, 0, 1, 0), (640, 2, 1, 0), (1000, 3, 2, 1), (4096, 4, 3, 0), (8192, 2, 5, 1),
    (8192, 100, 7, 0), (20000, 1, 160, 0),
])
def test_dilated_mask_matches_oracle(lib, N, window, dilation, causal):
    import numpy as np
    import attn_fwd_gb300.fa as fa
    import oracle
    got = fa.fa_block_mask_dilated(N, window, dilation, causal).numpy()
    np.testing.assert_array_equal(got, oracle.dilated_block_mask(N, window, dilation, bool(causal)))


def test_mask_generators_reject_bad_arguments(lib):
    buf = ctypes.create_string_buffer(16)
    assert lib.fa_block_mask_window(NULL, 128, 1, 1) == -1
    assert lib.fa_block_mask_window(buf, 0, 1, 1) == -1
    assert lib.fa_block_mask_window(buf, 128, -1, 1) == -1
    assert lib.fa_block_mask_dilated(buf, 128, 1, 0, 0) == -1
    assert lib.fa_block_mask_dilated(buf, 128, -1, 1, 0) == -1
    assert lib.fa_block_mask_window(buf, 1024 * 128 + 1, 1, 1) == -2


def test_decode_workspace_and_validation(lib):
    import attn_fwd_gb300.fa as fa
    assert fa.fa_decode_workspace_bytes(1, 1, 1, 64, 128) == 0          # one chunk: no workspace
    n = fa.fa_decode_workspace_bytes(8, 32, 1, 32768, 128)
    assert n > 0 and n % 256 == 0
    assert fa.fa_decode_workspace_bytes(1, 1, 9, 1024, 128) == 0         # Nq > 8 unsupported
    assert fa.fa_decode_workspace_bytes(1, 1, 1, 1024, 96) == 0
    sl = ctypes.c_void_p(4096 + 2)                                      # not 4-byte aligned
    assert lib.fa_decode(NULL, P, P, P, P, NULL, 1, 1, 1, 64, 128, 0.1, 0, NULL, NULL) == -1
    assert lib.fa_decode(P, P, P, P, P, sl, 1, 1, 1, 64, 128, 0.1, 0, NULL, NULL) == -1
    assert lib.fa_decode(P, P, P, P, P, NULL, 1, 1, 9, 64, 128, 0.1, 0, NULL, NULL) == -2
    assert lib.fa_decode(P, P, P, P, P, NULL, 1, 1, 0, 64, 128, 0.1, 0, NULL, NULL) == -1
    assert lib.fa_decode(P, P, P, P, P, NULL, 1, 1, 1, 64, 128, -1.0, 0, NULL, NULL) == -1
    # several chunks need a workspace
    assert lib.fa_decode(P, P, P, P, P, NULL, 8, 32, 1, 32768, 128, 0.1, 0, NULL, NULL) == -1


def test_dropout_argument_checks(lib):
    # dropout probability outside [0, 1) or not finite
    for pdrop in (-0.1, 1.0, float("nan")):
        assert lib.fa_fwd_dropout(P, P, P, P, P, NULL, 1, 1, 128, 64, 0.125, 0, pdrop, 1, NULL) == -1
        assert lib.fa_bwd_dropout(P, P, P, P, P, P, NULL, P, P, P, P, 1, 1, 128, 64, 0.125, 0, pdrop, 1, NULL) == -1
        assert lib.fa_bwd_main(P, P, P, P, NULL, P, P, P, 1, 1, 128, 64, 0.125, 0, pdrop, 1, NULL) == -1
    assert lib.fa_fwd_dropout(NULL, P, P, P, P, NULL, 1, 1, 128, 64, 0.125, 0, 0.1, 1, NULL) == -1


def test_dropout_effective_probability(lib):
    """The applied drop probability is the requested one rounded to a multiple
    of 1/256, as the oracle's dropout threshold defines it."""
    import attn_fwd_gb300.fa as fa
    import oracle
    for p in (0.0, 0.1, 0.25, 0.3, 0.5, 0.999, 1e-4, 0.998):
        assert fa.fa_dropout_effective_p(p) == oracle.dropout_threshold(p) / 256.0
    assert fa.fa_dropout_effective_p(0.1) == 26 / 256
    for bad in (-0.1, 1.0, float("nan")):
        assert lib.fa_dropout_effective_p(bad) == -1.0


def test_fp8_workspace_and_validation(lib):
    import attn_fwd_gb300.fa as fa
    assert fa.fa_fwd_fp8_workspace_bytes(2, 3, 300, 128) == 2 * 3 * 128 * 304 + (256 - (2 * 3 * 128 * 304) % 256) % 256
    assert fa.fa_fwd_fp8_workspace_bytes(1, 1, 128, 64) == 0          # d must be 128
    assert lib.fa_fwd_fp8(P, P, P, P, P, NULL, NULL, NULL, 1, 1, 128, 64, 0.1, 0, P, NULL) == -2
    assert lib.fa_fwd_fp8(P, P, P, P, P, NULL, NULL, NULL, 1, 1, 128, 128, 0.1, 0, NULL, NULL) == -1
    assert lib.fa_fwd_fp8(P, P, P, P, P, ctypes.c_void_p(4096 + 2), NULL, NULL, 1, 1, 128, 128, 0.1, 0, P, NULL) == -1
    assert lib.fa_fwd_fp8(P, P, P, P, P, NULL, NULL, NULL, 1, 1, 128, 128, 0.0, 0, P, NULL) == -1
