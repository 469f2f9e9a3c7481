"""Seeded synthetic inputs for exact attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both sides of every comparison (the CUDA path and the
CPU oracle) take their inputs from here, so neither ever computes the other's
inputs.

Recipe (the plainest reading of the workloads the pages and their benchmark
configurations describe):

* A CPU ``torch.Generator`` is seeded with the workload's seed.
* ``randn`` is drawn in fp32 in the order Q, K, V, dO, each of shape
  [B, H, N, d]; a workload with an amplitude multiplies the fp32 draws by it
  (peaked softmax rows); every tensor is then rounded to bf16.
* The oracle up-casts the *same* bf16 values to fp64.
* A block-sparse workload draws its mask from a fresh generator seeded with the
  same seed: ``rand(nb, nb) < p`` per 128x128 block, then every diagonal block
  is switched on.  One mask is shared by all (batch, head) pairs.
* A sliding-window workload's mask is a band of 128x128 blocks: query block i
  keeps key blocks i - left .. i + right (no random draw).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

BLOCK = 128  # granularity of the block-sparse mask (one bit per 128x128 block)


@dataclass(frozen=True)
class Workload:
    """One synthetic attention problem: sizes, mask kind and RNG recipe."""

    name: str
    B: int
    H: int
    N: int
    d: int
    seed: int
    causal: bool = False
    backward: bool = True
    amplitude: float = 1.0
    block_sparse_p: float | None = None  # keep-probability of an off-diagonal block
    window: tuple[int, int] | None = None  # (left, right) extent of a block band
    dropout_p: float = 0.0                 # dropout on P (mask seed = the workload's seed)
    fp8: bool = False                      # e4m3 inputs with per-head descales (forward only)
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    @property
    def mask_kind(self) -> str:
        if self.window is not None:
            return "causal+window" if self.causal else "window"
        if self.block_sparse_p is not None:
            return "causal+block" if self.causal else "block"
        return "causal" if self.causal else "none"


# The five benchmark workloads of this attention path.
WORKLOADS = {
    "fwd_b1h1n128d64": Workload(
        "fwd_b1h1n128d64", 1, 1, 128, 64, seed=0, backward=False,
        note="forward only, one 128x64 tile; latency case"),
    "fwdbwd_b4h8n1024d64": Workload(
        "fwdbwd_b4h8n1024d64", 4, 8, 1024, 64, seed=1,
        note="forward + backward, non-causal"),
    "fwdbwd_b2h16n4096d128_causal": Workload(
        "fwdbwd_b2h16n4096d128_causal", 2, 16, 4096, 128, seed=2, causal=True,
        note="forward + backward, causal, fully masked KV blocks skipped"),
    "fwd_b1h32n16384d128_causal_x3": Workload(
        "fwd_b1h32n16384d128_causal_x3", 1, 32, 16384, 128, seed=3, causal=True,
        backward=False, amplitude=3.0,
        note="forward only, causal, inputs x3 (peaked rows stress the rescale)"),
    "fwdbwd_b1h16n8192d128_blocksparse": Workload(
        "fwdbwd_b1h16n8192d128_blocksparse", 1, 16, 8192, 128, seed=4,
        block_sparse_p=0.25,
        note="forward + backward, 128x128 block mask, p=0.25 + diagonal"),
    # beyond the five: the headline shape with dropout 0.1 on P
    "fwdbwd_b2h16n4096d128_causal_dropout": Workload(
        "fwdbwd_b2h16n4096d128_causal_dropout", 2, 16, 4096, 128, seed=2, causal=True, dropout_p=0.1,
        note="forward + backward, causal, dropout 0.1 with regenerated masks"),
    # the headline shape's forward with 8-bit (e4m3) Q, K, V
    "fwd_b2h16n4096d128_causal_fp8": Workload(
        "fwd_b2h16n4096d128_causal_fp8", 2, 16, 4096, 128, seed=2, causal=True, backward=False, fp8=True,
        note="forward only, causal, e4m3 inputs with per-(batch, head) descales"),
    # a causal sliding window of 2048 keys (16 blocks)
    "fwdbwd_b1h16n16384d128_causal_window2k": Workload(
        "fwdbwd_b1h16n16384d128_causal_window2k", 1, 16, 16384, 128, seed=5, causal=True,
        window=(15, 0),
        note="forward + backward, causal, sliding window of 16 key blocks"),
}


@dataclass(frozen=True)
class DecodeWorkload:
    """The newest nq query tokens of each (batch, head) against a key/value
    cache of capacity N; `ragged` draws each batch's valid length uniformly
    from [N/4, N] (else every cache is full)."""

    name: str
    B: int
    H: int
    nq: int
    N: int
    d: int
    seed: int
    causal: bool = False
    ragged: bool = False
    note: str = field(default="", compare=False)
    backward: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    @property
    def mask_kind(self) -> str:
        return "causal" if self.causal else "none"


DECODE_WORKLOADS = {
    "decode_b8h32q1n32768d128": DecodeWorkload(
        "decode_b8h32q1n32768d128", 8, 32, 1, 32768, 128, seed=6,
        note="one new token per sequence, full 32k caches"),
    "decode_b16h32q1n8192d128_ragged": DecodeWorkload(
        "decode_b16h32q1n8192d128_ragged", 16, 32, 1, 8192, 128, seed=7, ragged=True,
        note="one new token, cache lengths uniform in [2k, 8k]"),
    "decode_b8h32q4n32768d128_causal": DecodeWorkload(
        "decode_b8h32q4n32768d128_causal", 8, 32, 4, 32768, 128, seed=8, causal=True,
        note="four new tokens (speculative decoding), causal among themselves"),
}


def make_decode_workload_inputs(w: DecodeWorkload) -> dict[str, torch.Tensor]:
    """q, k, v (CPU bf16) and seqlens (CPU int32 [B]) of a decode workload."""
    t = make_decode_inputs(w.B, w.H, w.nq, w.N, w.d, w.seed)
    if w.ragged:
        g = torch.Generator(device="cpu").manual_seed(w.seed + 1)
        t["seqlens"] = torch.randint(w.N // 4, w.N + 1, (w.B,), generator=g, dtype=torch.int32)
    else:
        t["seqlens"] = torch.full((w.B,), w.N, dtype=torch.int32)
    return t


def make_qkvdo(B: int, H: int, N: int, d: int, seed: int, amplitude: float = 1.0,
               with_dout: bool = True) -> dict[str, torch.Tensor]:
    """Draw Q, K, V (and dO) as CPU bf16 tensors of shape [B, H, N, d]."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    names = ["q", "k", "v"] + (["do"] if with_dout else [])
    out = {}
    for nm in names:
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        if amplitude != 1.0:
            x = x * amplitude
        out[nm] = x.to(torch.bfloat16)
    return out


def make_decode_inputs(B: int, H: int, Nq: int, Nk: int, d: int, seed: int) -> dict[str, torch.Tensor]:
    """Decoding inputs as CPU bf16 tensors: q [B, H, Nq, d] (the newest tokens)
    and the cache k, v [B, H, Nk, d], drawn in that order from one generator."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    out = {"q": torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)}
    for nm in ("k", "v"):
        out[nm] = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_fp8_inputs(B: int, H: int, N: int, d: int, seed: int) -> dict[str, torch.Tensor]:
    """8-bit inputs: Q, K, V drawn as for make_qkvdo (fp32 randn in that order),
    then each (batch, head) of each tensor stored as e4m3 after division by
    its descale amax / 448 (so it fills the e4m3 range).  Returns q8, k8, v8
    (float8_e4m3fn, CPU) and qd, kd, vd (fp32 [B, H])."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    out = {}
    for nm in ("q", "k", "v"):
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        ds = x.abs().amax(dim=(2, 3)) / 448.0
        out[nm + "8"] = (x / ds[..., None, None]).to(torch.float8_e4m3fn)
        out[nm + "d"] = ds.contiguous()
    return out


def make_block_mask(N: int, seed: int, p: float, block: int = BLOCK) -> torch.Tensor:
    """Block mask as uint8 [N/block, N/block]; diagonal blocks are always kept."""
    if N % block:
        raise ValueError("N must be a multiple of the block size")
    nb = N // block
    g = torch.Generator(device="cpu").manual_seed(seed)
    keep = (torch.rand((nb, nb), generator=g) < p).to(torch.uint8)
    keep.fill_diagonal_(1)
    return keep


def make_window_mask(N: int, left: int, right: int, block: int = BLOCK) -> torch.Tensor:
    """Band of blocks as uint8 [nb, nb]: query block i keeps i - left .. i + right."""
    nb = -(-N // block)
    return torch.ones((nb, nb), dtype=torch.uint8).tril(right).triu(-left).contiguous()


def make_workload_inputs(w: Workload, heads: slice | None = None) -> dict[str, torch.Tensor]:
    """All inputs of a workload (CPU).  ``heads`` optionally keeps a head slice."""
    if w.fp8:
        t = make_fp8_inputs(w.B, w.H, w.N, w.d, w.seed)
    else:
        t = make_qkvdo(w.B, w.H, w.N, w.d, w.seed, w.amplitude, with_dout=w.backward)
    if heads is not None:
        t = {k: v[:, heads].contiguous() for k, v in t.items()}
    if w.block_sparse_p is not None:
        t["block_mask"] = make_block_mask(w.N, w.seed, w.block_sparse_p)
    if w.window is not None:
        t["block_mask"] = make_window_mask(w.N, *w.window)
    return t
