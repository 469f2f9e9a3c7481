"""Plain, slow, fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and its reference arm) may import this package.  The CUDA library never
reaches it, and it shares no code with the CUDA path.

Pages cited below (by title and section):

* [P1] "【多模态大模型】FlashAttention in NeurIPS 2022" (coreui.cn), section
  "2.1 拆分": safe softmax with m(s), l(s), the m / l / o update rules and the
  worked example softmax([1,2,3,10]) with V=[[1,2],[3,4],[5,6],[7,8]].
* [P2] "FlashAttention" notes (maosong.website): "Standard Attention
  Implementation" (S=QK^T, P=softmax(S), O=PV), "Tiling" (merge of m and l),
  "Correctness" (Theorem 1), "Backward Pass of flashattention" (dV, dP, D_i,
  dS, dq_i, dk_j), "Block-sparse Flashattention" (mask M, S restricted by M).
* [P3] "Transformer 入门" (cansult.github.io), section "flash attention":
  S = QK^T / sqrt(d), m = rowmax(S), l = rowsum(exp(S - m)), tiles T_r, T_c.
* [P4] "Как работает FlashAttention математически" (aivaro.ru), sections 3
  (online softmax), 4 (output correction), 6 (per-block pseudocode), and the
  practice exercise (tiled vs standard within 1e-5).

Readings where the pages are silent or disagree (each also listed in the design
notes):

* Scale: S = scale * Q K^T with scale = 1/sqrt(d) [P3]; [P1] drops the factor.
  The backward carries it to dQ and dK by the chain rule.
* Masked entries are -inf (they add nothing to m, l or O); [P2]'s block-sparse
  text writes 0, which would not skip anything.
* Causal: key j is visible to query i iff j <= i (equal query/key lengths).
* Block-sparse: mask[i // block, j // block] keeps or drops a whole block;
  causal and a block mask together keep what both keep.
* Sliding-window and dilated patterns are block masks (one bit per block),
  the granularity at which the pages place them under block-sparse attention;
  dilated: key block i + t * dilation for |t| <= window.
* A row with no visible key gets O = 0, LSE = -inf and zero gradients.
* LSE = m + ln(l), natural log.

Everything here works on float64 arrays laid out [B, H, N, d] (V may have its
own last dimension).  Parity status: every public function is pinned by the
CPU tests (worked example, closed forms, invariants, finite differences, and
PyTorch's own fp64 attention routine).
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------- #
# masks
# --------------------------------------------------------------------------- #
def visible(nq: int, nk: int, causal: bool = False, block_mask=None,
            block: int = 128, rows=None) -> np.ndarray:
    """Boolean [len(rows), nk]: True where query row i may attend to key j.

    Causal: j <= i.  Block-sparse [P2 "Block-sparse Flashattention"]: the
    N x N mask M is given at block granularity, M[i, j] = mask[i//block, j//block].
    """
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    cols = np.arange(nk)
    vis = np.ones((rows.size, nk), dtype=bool)
    if causal:
        vis &= cols[None, :] <= rows[:, None]
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        vis &= bm[rows[:, None] // block, cols[None, :] // block]
    return vis


def window_block_mask(N: int, left: int, right: int, block: int = 128) -> np.ndarray:
    """Sliding window at block granularity, uint8 [nb, nb], nb = ceil(N / block).

    ["Как работает FlashAttention математически" section 9: block-sparse
    FlashAttention serves sliding-window patterns.]  Query block i keeps the
    key blocks i - left, ..., i + right that exist.
    """
    nb = -(-N // block)
    m = np.zeros((nb, nb), dtype=np.uint8)
    for i in range(nb):
        for j in range(max(0, i - left), min(nb, i + right + 1)):
            m[i, j] = 1
    return m


def dilated_block_mask(N: int, window: int, dilation: int, causal: bool = False,
                       block: int = 128) -> np.ndarray:
    """Dilated window at block granularity, uint8 [nb, nb].

    [Same section: dilated attention as a block-sparse pattern.]  Query block i
    keeps key blocks i + t * dilation for t = -window .. window (t <= 0 when
    causal), those that exist.
    """
    nb = -(-N // block)
    m = np.zeros((nb, nb), dtype=np.uint8)
    for i in range(nb):
        for t in range(-window, (0 if causal else window) + 1):
            j = i + t * dilation
            if 0 <= j < nb:
                m[i, j] = 1
    return m


# --------------------------------------------------------------------------- #
# the definition: materialised S and P per (batch, head)
# --------------------------------------------------------------------------- #
def _scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * q k^T for one head [P3 "flash attention" definitions]."""
    return scale * (q @ k.T)


def _apply_mask(s: np.ndarray, vis: np.ndarray) -> np.ndarray:
    """Masked entries become -inf so they add nothing to m, l or O."""
    return np.where(vis, s, NEG_INF)


def _row_softmax(s: np.ndarray):
    """Safe softmax per row [P1 2.1; P2 "Tiling"]: m = max, f = exp(s - m),
    l = sum f, P = f / l.  Returns (P, m, l); an all -inf row gives P = 0."""
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    f = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 on masked entries
    l = f.sum(axis=1)
    l_safe = np.where(l > 0, l, 1.0)
    p = f / l_safe[:, None]
    return p, m, l


def _lse(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """LSE = m + ln(l); -inf for a row without visible keys."""
    with np.errstate(divide="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)


def head_probs(q, k, scale, causal=False, block_mask=None, block=128, rows=None):
    """P (rows x N) and LSE (rows) of one head, materialised."""
    s = _scores(q if rows is None else q[np.asarray(rows)], k, scale)
    s = _apply_mask(s, visible(q.shape[0], k.shape[0], causal, block_mask, block, rows))
    p, m, l = _row_softmax(s)
    return p, _lse(m, l)


def forward(q, k, v, scale, causal=False, block_mask=None, block=128,
            row_chunk: int | None = None):
    """O = softmax(S) V and LSE for [B, H, N, d] fp64 inputs
    [P2 "Standard Attention Implementation"; P3 definitions with the scale].

    ``row_chunk`` splits the query rows of a head into chunks of full rows, so
    a long sequence never holds all of S at once; each row's softmax is still
    the plain definition over the whole row.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, N, _ = q.shape
    o = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse = np.zeros((B, H, N))
    step = N if row_chunk is None else row_chunk
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, step):
                rows = np.arange(r0, min(N, r0 + step))
                p, lse_r = head_probs(q[b, h], k[b, h], scale, causal, block_mask,
                                      block, rows if step != N else None)
                o[b, h, rows] = p @ v[b, h]
                lse[b, h, rows] = lse_r
    return o, lse


def forward_rows(q, k, v, scale, b, h, rows, causal=False, block_mask=None, block=128,
                 dropout_p: float = 0.0, seed: int = 0):
    """O and LSE of selected query rows of head (b, h) only: for sampled checks
    of workloads too large to materialise.  With dropout_p, the rows of
    forward_dropout."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q[b, h], k[b, h], v[b, h]))
    p, lse = head_probs(q, k, scale, causal, block_mask, block, rows)
    if dropout_p:
        p = p * dropout_keep(b, h, rows, np.arange(k.shape[0]), dropout_p, seed) * (
            256.0 / (256 - dropout_threshold(dropout_p)))
    return p @ v, lse


def _softmax_backward(p: np.ndarray, dp: np.ndarray, d_row: np.ndarray) -> np.ndarray:
    """dS_ij = P_ij (dP_ij - D_i) [P2 "Backward Pass of flashattention"]."""
    return p * (dp - d_row[:, None])


def backward(q, k, v, do, scale, causal=False, block_mask=None, block=128):
    """dQ, dK, dV and D for [B, H, N, d] fp64 inputs, using the oracle's own O and P.

    Follows [P2 "Backward Pass of flashattention"] with the scale's chain rule:
    dV = P^T dO;  dP = dO V^T;  D_i = sum_j P_ij dP_ij;  dS = P o (dP - D);
    dQ = scale * dS K;  dK = scale * dS^T Q.
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    B, H, N, _ = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dvec = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            p, _ = head_probs(q[b, h], k[b, h], scale, causal, block_mask, block)
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            d_row = (p * dp).sum(axis=1)
            ds = _softmax_backward(p, dp, d_row)
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
            dvec[b, h] = d_row
    return dq, dk, dv, dvec


def backward_rows_dq(q, k, v, do, scale, b, h, rows, causal=False, block_mask=None,
                     block=128):
    """dQ of selected query rows of head (b, h) [P2: dq_i = sum_j P_ij (dP_ij - D_i) k_j],
    with D_i taken as do_i . o_i of the oracle's own o_i."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q[b, h], k[b, h], v[b, h], do[b, h]))
    rows = np.asarray(rows)
    p, _ = head_probs(q, k, scale, causal, block_mask, block, rows)
    o = p @ v
    dp = do[rows] @ v.T
    d_row = (do[rows] * o).sum(axis=1)
    return scale * (_softmax_backward(p, dp, d_row) @ k)


def backward_rows(q, k, v, do, scale, b, h, rows, causal=False, block_mask=None, block=128,
                  dropout_p: float = 0.0, seed: int = 0):
    """The backward restricted to selected query rows of head (b, h): dQ of
    those rows and their contributions to dK and dV [P2 "Backward Pass of
    flashattention": dv_j = sum_i P_ij do_i, dk_j = sum_i dS_ij q_i, both sums
    over query rows i, so a partition of the rows splits them exactly].  With
    dropout_p, the rows of backward_dropout.
    Returns (dq_rows, dk_part, dv_part, o_rows, lse_rows)."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q[b, h], k[b, h], v[b, h], do[b, h]))
    rows = np.asarray(rows)
    p, lse = head_probs(q, k, scale, causal, block_mask, block, rows)
    zc = 1.0
    if dropout_p:
        zc = dropout_keep(b, h, rows, np.arange(k.shape[0]), dropout_p, seed) * (
            256.0 / (256 - dropout_threshold(dropout_p)))
    o = (p * zc) @ v
    dp = (do[rows] @ v.T) * zc
    d_row = (p * dp).sum(axis=1)
    ds = _softmax_backward(p, dp, d_row)
    return scale * (ds @ k), scale * (ds.T @ q[rows]), (p * zc).T @ do[rows], o, lse


# --------------------------------------------------------------------------- #
# the tiled algorithm, step by step as the pages state it
# --------------------------------------------------------------------------- #
def tiled_forward(q, k, v, scale, Br: int, Bc: int, causal=False, block_mask=None,
                  block=128, trace=False):
    """Tiled forward with the online-softmax recurrence, one head at a time.

    For each query tile Q_i (B_r rows) [P3 tiles T_r, T_c; V2 loop order]:
    m = -inf, l = 0, O = 0; then for each key/value tile K_j, V_j (B_c rows)
    [P4 section 6 pseudocode; P1 2.1 update rules]:
        S_ij   = scale * Q_i K_j^T  (masked entries -inf)
        m_new  = max(m, rowmax(S_ij))
        l_new  = exp(m - m_new) l + rowsum(exp(S_ij - m_new))
        O      = (l exp(m - m_new) O + exp(S_ij - m_new) V_j) / l_new
        m, l   = m_new, l_new
    and finally LSE = m + ln l.  Rows whose running max is still -inf skip the
    update (nothing visible yet).  With ``trace`` it also returns, per head and
    query tile, the (m, l, O) after every key tile.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, N, _ = q.shape
    Nk = k.shape[2]
    o_all = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse_all = np.zeros((B, H, N))
    traces = []
    for b in range(B):
        for h in range(H):
            for i0 in range(0, N, Br):
                rows = np.arange(i0, min(N, i0 + Br))
                m = np.full(rows.size, NEG_INF)
                l = np.zeros(rows.size)
                o = np.zeros((rows.size, v.shape[-1]))
                tr = []
                for j0 in range(0, Nk, Bc):
                    cols = np.arange(j0, min(Nk, j0 + Bc))
                    s = scale * (q[b, h, rows] @ k[b, h, cols].T)
                    vis = visible(N, Nk, causal, block_mask, block, rows)[:, cols]
                    s = np.where(vis, s, NEG_INF)
                    m_new = np.maximum(m, s.max(axis=1))
                    live = np.isfinite(m_new)
                    mn = np.where(live, m_new, 0.0)
                    alpha = np.where(live, np.exp(np.where(live, m, 0.0) - mn), 0.0)
                    alpha = np.where(np.isfinite(m), alpha, 0.0)   # exp(-inf - m_new) = 0
                    pt = np.exp(s - mn[:, None])
                    l_new = alpha * l + pt.sum(axis=1)
                    num = (l * alpha)[:, None] * o + pt @ v[b, h, cols]
                    o = np.where(live[:, None], num / np.where(live, l_new, 1.0)[:, None], 0.0)
                    m, l = np.where(live, m_new, NEG_INF), np.where(live, l_new, 0.0)
                    if trace:
                        tr.append((m.copy(), l.copy(), o.copy()))
                o_all[b, h, rows] = o
                lse_all[b, h, rows] = _lse(m, l)
                if trace:
                    traces.append(tr)
    if trace:
        return o_all, lse_all, traces
    return o_all, lse_all


# --------------------------------------------------------------------------- #
# dropout with regenerated masks
# --------------------------------------------------------------------------- #
# The pages keep only O(N) statistics and regenerate the random dropout masks
# in the backward instead of storing them ("Как работает FlashAttention
# математически", section 5; "FlashAttention" notes, "Backward Pass of
# flashattention").  They name no generator; the reading here: the
# counter-based generator Philox4x32-10 of Salmon, Moraes, Dror and Shaw,
# "Parallel random numbers: as easy as 1, 2, 3" (SC'11), key = the 64-bit
# seed, counter = (j // 4, i // 4, h, b) for query i and key j, so one call
# covers a 4 x 4 block; element (i, j) takes byte j % 4 (little-endian) of
# output word i % 4 and is kept iff that byte >= t = round(256 p), t <= 255;
# kept entries are scaled by 256 / (256 - t).

_PHILOX_M = (0xD2511F53, 0xCD9E8D57)        # round multipliers
_PHILOX_W = (0x9E3779B9, 0xBB67AE85)        # key increments (Weyl sequence)


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds on uint32 counters [..., 4] and a key (k0, k1):
    each round multiplies words 0 and 2 by the two constants, and the new
    words are (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0));
    the key advances by the Weyl increments between rounds."""
    c = np.array(ctr, dtype=np.uint64) & 0xFFFFFFFF
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    mask = np.uint64(0xFFFFFFFF)
    for r in range(10):
        if r:
            k0 = (k0 + _PHILOX_W[0]) & 0xFFFFFFFF
            k1 = (k1 + _PHILOX_W[1]) & 0xFFFFFFFF
        p0 = c[..., 0] * np.uint64(_PHILOX_M[0])
        p1 = c[..., 2] * np.uint64(_PHILOX_M[1])
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        c = np.stack([hi1 ^ c[..., 1] ^ np.uint64(k0), lo1, hi0 ^ c[..., 3] ^ np.uint64(k1), lo0], axis=-1)
    return c.astype(np.uint32)


def dropout_threshold(p: float) -> int:
    """Byte threshold t = round(256 p), at most 255: a byte below t drops."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(255, int(np.floor(256.0 * p + 0.5)))


def dropout_bytes(b: int, h: int, rows, cols, seed: int) -> np.ndarray:
    """uint8 [len(rows), len(cols)]: the random byte of each (query, key) pair
    of head (b, h): byte j % 4 of word i % 4 of Philox(counter (j//4, i//4, h, b))."""
    rows, cols = np.asarray(rows, dtype=np.int64), np.asarray(cols, dtype=np.int64)
    # one generator call per 4 x 4 block that the pairs touch
    rb, ri = np.unique(rows // 4, return_inverse=True)
    cb, ci = np.unique(cols // 4, return_inverse=True)
    gr, gc = np.meshgrid(rb, cb, indexing="ij")
    ctr = np.stack([gc, gr, np.full_like(gr, h), np.full_like(gr, b)], axis=-1)
    words = philox4x32_10(ctr, (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))   # [blocks_i, blocks_j, 4]
    word = words[ri[:, None], ci[None, :], (rows % 4)[:, None]]
    return ((word >> (8 * (cols % 4))[None, :].astype(np.uint32)) & 0xFF).astype(np.uint8)


def dropout_keep(b: int, h: int, rows, cols, p: float, seed: int) -> np.ndarray:
    """Boolean [len(rows), len(cols)]: which (query, key) pairs of head (b, h)
    dropout keeps (random byte >= round(256 p))."""
    return dropout_bytes(b, h, rows, cols, seed) >= dropout_threshold(p)


def forward_dropout(q, k, v, scale, p: float, seed: int, causal=False, block_mask=None, block=128,
                    b0: int = 0, h0: int = 0):
    """O = (P o Z) V * 256 / (256 - t) with P the plain softmax and Z the
    regenerated keep mask; LSE is that of P (dropout acts after the softmax).
    Input head (b, h) is head (b0 + b, h0 + h) of the whole problem (the mask
    depends on it)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, N, _ = q.shape
    Nk = k.shape[2]
    inv_keep = 256.0 / (256 - dropout_threshold(p))
    o = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            pr, lse[b, h] = head_probs(q[b, h], k[b, h], scale, causal, block_mask, block)
            z = dropout_keep(b0 + b, h0 + h, np.arange(N), np.arange(Nk), p, seed)
            o[b, h] = (pr * z * inv_keep) @ v[b, h]
    return o, lse


def backward_dropout(q, k, v, do, scale, p: float, seed: int, causal=False, block_mask=None, block=128,
                     b0: int = 0, h0: int = 0):
    """Gradients of forward_dropout ["FlashAttention" notes, "Backward Pass of
    flashattention", with the dropped probabilities P~ = P o Z * c]:
    dV = P~^T dO;  dP = (dO V^T) o Z * c;  D_i = sum_j P_ij dP_ij;
    dS = P o (dP - D);  dQ = scale * dS K;  dK = scale * dS^T Q."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    B, H, N, _ = q.shape
    Nk = k.shape[2]
    inv_keep = 256.0 / (256 - dropout_threshold(p))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dvec = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            pr, _ = head_probs(q[b, h], k[b, h], scale, causal, block_mask, block)
            zc = dropout_keep(b0 + b, h0 + h, np.arange(N), np.arange(Nk), p, seed) * inv_keep
            dv[b, h] = (pr * zc).T @ do[b, h]
            dp = (do[b, h] @ v[b, h].T) * zc
            d_row = (pr * dp).sum(axis=1)
            ds = _softmax_backward(pr, dp, d_row)
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
            dvec[b, h] = d_row
    return dq, dk, dv, dvec


# --------------------------------------------------------------------------- #
# 8-bit (e4m3) inputs
# --------------------------------------------------------------------------- #
# The pages name 8-bit tensor-core arithmetic only as the FlashAttention-3
# extension ("Как работает FlashAttention математически", section 9).  The
# reading here: inputs are e4m3 bytes with per-(batch, head) descale factors,
# the real input is byte value x descale, and the result to reproduce is exact
# attention on those real inputs; the kernel's rounding of P to e4m3 is an
# approximation whose error fp8_error_model bounds.

def e4m3_decode(codes) -> np.ndarray:
    """Value of e4m3 bytes (1 sign bit, 4 exponent bits with bias 7, 3
    mantissa bits; exponent 0 is subnormal: m/8 * 2^-6; no infinities; the
    codes 0x7F and 0xFF are NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def forward_fp8(q8, k8, v8, q_descale, k_descale, v_descale, scale, causal=False):
    """Exact attention on the real inputs q8 dq, k8 dk, v8 dv (q8, k8, v8: e4m3
    bytes [B, H, N, d] as uint8; descales [B, H]).  Returns (O, LSE, P) with P
    the per-head probabilities [B, H, N, N] (for the error model)."""
    dq, dk, dv = (np.asarray(x, dtype=np.float64)[..., None, None] for x in (q_descale, k_descale, v_descale))
    q, k, v = e4m3_decode(q8) * dq, e4m3_decode(k8) * dk, e4m3_decode(v8) * dv
    B, H, N, _ = q.shape
    o, lse = forward(q, k, v, scale, causal=causal)
    probs = np.zeros((B, H, N, k.shape[2]))
    for b in range(B):
        for h in range(H):
            probs[b, h], _ = head_probs(q[b, h], k[b, h], scale, causal)
    return o, lse, probs, v


def fp8_error_model(o, probs, v, rel: float = 2.0 ** -4, row_chunk: int = 64):
    """Effect on O of rounding every attention weight to e4m3 (relative error
    d_j at most `rel`: 3 mantissa bits) while O is still divided by the exact
    row sum: O' - O = sum_j w_j d_j v_j.  Weights below 2^-14 of the row's
    largest are flushed or rounded with an absolute error up to 2^-14 of it
    (e4m3's subnormal step against a row maximum of at least 16).
    Returns (bound, sigma): the worst case rel * sum_j w_j |v_j| + n 2^-14
    max_j |v_j|, and the standard deviation when the d_j are independent and
    uniform on [-rel, rel]: rel / sqrt(3) * sqrt(sum_j w_j^2 v_j^2).  Rows are
    taken in chunks."""
    B, H, N, d = o.shape
    bound = np.zeros_like(o)
    sigma = np.zeros_like(o)
    for b in range(B):
        for h in range(H):
            av = np.abs(v[b, h])
            for r0 in range(0, N, row_chunk):
                rows = slice(r0, min(N, r0 + row_chunk))
                w = probs[b, h, rows]                                    # [r, Nk]
                n_vis = (w > 0).sum(axis=1)[:, None]
                vis_max = np.stack([av[w[i] > 0].max(axis=0) if n_vis[i, 0] else np.zeros(d)
                                    for i in range(w.shape[0])])
                bound[b, h, rows] = rel * (w @ av) + n_vis * 2.0 ** -14 * vis_max
                sigma[b, h, rows] = rel / np.sqrt(3.0) * np.sqrt((w ** 2) @ (v[b, h] ** 2))
    return bound, sigma


# --------------------------------------------------------------------------- #
# decoding: the newest query tokens against a cache of keys and values
# --------------------------------------------------------------------------- #
def decode_visible(nq: int, L: int, causal: bool = False) -> np.ndarray:
    """Boolean [nq, L]: which of the L cached keys each of the nq newest query
    tokens may attend to.  Query i sits at sequence position L - nq + i; with
    the causal mask it sees keys 0 .. L - nq + i, else all L."""
    vis = np.ones((nq, L), dtype=bool)
    if causal:
        pos = L - nq + np.arange(nq)
        vis &= np.arange(L)[None, :] <= pos[:, None]
    return vis


def decode(q, k, v, scale, seqlens=None, causal=False):
    """O and LSE of q [B, H, Nq, d] against a cache k, v [B, H, Nk, d] whose
    first seqlens[b] rows are valid (all Nk without seqlens), materialised
    ["Как работает FlashAttention математически" section 9: FlashDecoding,
    K and V cached, Q the newest token(s); the softmax is the plain definition
    of "FlashAttention" notes, "Standard Attention Implementation"]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, nq, _ = q.shape
    o = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse = np.full((B, H, nq), NEG_INF)
    for b in range(B):
        L = k.shape[2] if seqlens is None else int(seqlens[b])
        if L == 0:
            continue
        for h in range(H):
            s = _apply_mask(_scores(q[b, h], k[b, h, :L], scale), decode_visible(nq, L, causal))
            p, m, l = _row_softmax(s)
            o[b, h] = p @ v[b, h, :L]
            lse[b, h] = _lse(m, l)
    return o, lse


def decode_split(q, k, v, scale, chunk: int, seqlens=None, causal=False):
    """The split-KV form of decode: each chunk of `chunk` cached keys gives its
    own normalised O_c and LSE_c (the plain softmax over that chunk); the
    chunks are merged with the statistics merge of "FlashAttention" notes,
    "Tiling" -- M = max_c LSE_c, w_c = exp(LSE_c - M), O = sum w_c O_c / sum w_c,
    LSE = M + ln(sum w_c).  Chunks with no visible key carry LSE_c = -inf."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, nq, _ = q.shape
    o = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse = np.full((B, H, nq), NEG_INF)
    for b in range(B):
        L = k.shape[2] if seqlens is None else int(seqlens[b])
        vis = decode_visible(nq, L, causal)
        for h in range(H):
            parts = []
            for c0 in range(0, L, chunk):
                cols = np.arange(c0, min(L, c0 + chunk))
                s = _apply_mask(_scores(q[b, h], k[b, h, cols], scale), vis[:, cols])
                p, m, l = _row_softmax(s)
                parts.append((p @ v[b, h, cols], _lse(m, l)))
            if not parts:
                continue
            lses = np.stack([pl for _, pl in parts])               # [chunks, nq]
            M = lses.max(axis=0)
            fin = np.isfinite(M)
            w = np.exp(lses - np.where(fin, M, 0.0)[None, :])      # exp(-inf) = 0
            W = w.sum(axis=0)
            acc = sum(wc[:, None] * oc for wc, (oc, _) in zip(w, parts))
            o[b, h] = np.where(fin[:, None], acc / np.where(fin, W, 1.0)[:, None], 0.0)
            lse[b, h] = np.where(fin, M + np.log(np.where(fin, W, 1.0)), NEG_INF)
    return o, lse


def merge_stats(m1, l1, m2, l2):
    """Merge (m, l) of two parts of a row [P2 "Tiling"]:
    m = max(m1, m2);  l = exp(m1 - m) l1 + exp(m2 - m) l2."""
    m = np.maximum(m1, m2)
    return m, np.exp(m1 - m) * l1 + np.exp(m2 - m) * l2


# --------------------------------------------------------------------------- #
# error scale of gradients computed with bf16 operands and fp32 sums
# --------------------------------------------------------------------------- #
BF16_U = 2.0 ** -8      # unit roundoff of bf16 (8 significant bits, round to nearest even)
FP32_STEP = 2.0 ** -23  # one fp32 rounding step, truncation included (24 significant bits)


def forward_error_bound(q, k, v, scale, causal=False, block_mask=None, block=128, row_chunk=None,
                        u: float = BF16_U, rows=None):
    """Worst-case effect on O of feeding the probabilities to the P V product
    as bf16, per element [B, H, N, dv].

    O_i = sum_j w_ij V_j with weights w = P (1 + e), |e_ij| <= u (u = 2^-8),
    divided by the sum of the rounded weights or by the exact one.  To first
    order the first moves O_i by sum_j P_ij e_ij (V_j - O_i), the second by
    sum_j P_ij e_ij V_j; both are at most u sum_j P_ij (|V_j| + |O_i|) =
    u ((P |V|)_i + |O_i|).  With bf16 inputs this rounding is unavoidable, and
    on peaked rows with large |V| (two keys of weight 1/2 whose V differ by
    20 move O by up to 2^-8 x 10) it exceeds a fixed 1e-2 on its own.  Query
    rows are taken in chunks of ``row_chunk`` full rows; with ``rows``, only
    those query rows (the result is then [B, H, len(rows), dv])."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, N, _ = q.shape
    sel = np.arange(N) if rows is None else np.asarray(rows)
    out = np.zeros((B, H, len(sel), v.shape[-1]))
    step = len(sel) if row_chunk is None else row_chunk
    for b in range(B):
        for h in range(H):
            av = np.abs(v[b, h])
            for r0 in range(0, len(sel), step):
                idx = np.arange(r0, min(len(sel), r0 + step))
                p, _ = head_probs(q[b, h], k[b, h], scale, causal, block_mask, block, sel[idx])
                out[b, h, idx] = u * (p @ av + np.abs(p @ v[b, h]))
    return out


def grad_error_model(q, k, v, do, scale, causal=False, block_mask=None, block=128,
                     row_chunk: int = 1024, u: float = BF16_U, f32: float = FP32_STEP):
    """Per-element error scale of dQ, dK, dV computed from bf16 inputs with
    bf16 outputs and fp32 accumulation.

    Where such an implementation must round to bf16: the forward stores O
    (and its P V product takes P as bf16); the backward's products take P
    (dV = P^T dO) and dS (dK = s dS^T Q, dQ = s dS K) as bf16, and
    D_i = dO_i . O_i uses the stored O ["FlashAttention" notes, "Backward Pass
    of flashattention": D_i = do_i^T o_i].  Rounding x to bf16 moves it by at
    most u |x|; taken as uniform, by a standard deviation of at most
    u |x| / sqrt(3).  To first order, with independent rounding errors e:

    * D_i: the forward's rounding of P moves O_i by sum_j P_ij e_ij (V_j - O_i)
      (row sum of the rounded weights) or sum_j P_ij e_ij V_j (exact sum), so
      D_i by sum_j P_ij e_ij (dP_ij - D_i) or sum_j P_ij e_ij dP_ij; O's own
      rounding adds sum_c dO_ic O_ic e_ic:
      Var D_i <= (u^2/3) [2 sum_j P_ij^2 (dP_ij^2 + D_i^2) + sum_c dO_ic^2 O_ic^2].
    * dS_ij, apart from D_i: Var <= (u^2/3) dS_ij^2.
    * dV_jc = sum_i P_ij dO_ic:  Var = (u^2/3) sum_i P_ij^2 dO_ic^2.
    * dK_jc = s sum_i dS_ij Q_ic:  Var = s^2 [sum_i Var(dS_ij) Q_ic^2 + sum_i P_ij^2 Q_ic^2 Var D_i].
    * dQ_ic = s sum_j dS_ij K_jc:  Var = s^2 [sum_j Var(dS_ij) K_jc^2 + (sum_j P_ij K_jc)^2 Var D_i]
      (D_i's error is shared by the whole row, so it adds coherently over j).

    fp32 effects, as worst cases added in quadrature: a product of length n
    summed in steps of 16 is off by at most (n/16 + 2) f32 times the sum of
    its absolute terms (f32 = 2^-23, one rounding or truncation step), which
    bounds the scores' error, so P's relative error, at
    (d/16 + 2) f32 s sum_c |Q_ic K_jc| + f32 (|LSE_i| + 8), dP's at
    (d/16 + 2) f32 sum_c |dO_ic V_jc| and D_i's at (d/16 + 2) f32
    sum_c |dO_ic O_ic|; each gradient's own sum over N terms is off by at
    most acc = (N/16 + N/128 + 2) f32 times the sum of its absolute terms
    (tensor-core steps of 16, then per-tile partial sums).

    Returns (sigma, acc), each a tuple (dQ, dK, dV) of arrays [B, H, N, d].
    A gradient g then satisfies |g - r| <= u |r| + (1 + u)(k sigma + acc) for
    the exact r and a few k; u |r| is the output's own rounding.  Query rows
    are taken in chunks of ``row_chunk`` full rows."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    B, H, N, d = q.shape
    r2 = u * u / 3.0
    cd = (d / 16.0 + 2.0) * f32
    n_acc = (N / 16.0 + N / 128.0 + 2.0) * f32
    sig = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)]
    acc = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)]
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = q[b, h], k[b, h], v[b, h], do[b, h]
            aq, ak, av = np.abs(qh), np.abs(kh), np.abs(vh)
            var_dk = np.zeros_like(kh)
            var_dv = np.zeros_like(vh)
            abs_dk = np.zeros_like(kh)
            abs_dv = np.zeros_like(vh)
            for r0 in range(0, N, row_chunk):
                rows = np.arange(r0, min(N, r0 + row_chunk))
                p, lse = head_probs(qh, kh, scale, causal, block_mask, block, rows)
                o = p @ vh
                dor = doh[rows]
                adr = np.abs(dor)
                dp = dor @ vh.T
                d_row = (dor * o).sum(axis=1)
                ds = _softmax_backward(p, dp, d_row)
                p2 = p * p
                lse_f = np.where(np.isfinite(lse), np.abs(lse), 0.0)
                rho = cd * scale * (np.abs(qh[rows]) @ ak.T) + f32 * (lse_f[:, None] + 8.0)
                var_d = (r2 * (2.0 * (p2 * (dp * dp + d_row[:, None] ** 2)).sum(axis=1) + ((dor * o) ** 2).sum(axis=1))
                         + ((p * rho * np.abs(dp - d_row[:, None])).sum(axis=1)) ** 2
                         + (cd * np.abs(dor * o).sum(axis=1)) ** 2)
                var_ds = r2 * ds * ds + (rho * ds) ** 2 + (p * cd * (adr @ av.T)) ** 2
                qr = qh[rows]
                var_dq = scale ** 2 * (var_ds @ (kh * kh) + (p @ kh) ** 2 * var_d[:, None])
                sig[0][b, h, rows] = np.sqrt(var_dq)
                acc[0][b, h, rows] = n_acc * scale * (np.abs(ds) @ ak)
                var_dk += scale ** 2 * (var_ds.T @ (qr * qr) + p2.T @ (qr * qr * var_d[:, None]))
                abs_dk += n_acc * scale * (np.abs(ds).T @ np.abs(qr))
                var_dv += r2 * (p2.T @ (dor * dor)) + ((p * rho) ** 2).T @ (dor * dor)
                abs_dv += n_acc * (p.T @ adr)
            sig[1][b, h], sig[2][b, h] = np.sqrt(var_dk), np.sqrt(var_dv)
            acc[1][b, h], acc[2][b, h] = abs_dk, abs_dv
    return tuple(sig), tuple(acc)
