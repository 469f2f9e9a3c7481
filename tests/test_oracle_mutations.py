"""Plant plausible mistakes in the oracle (on the CPU) and require that at least
one pin fails for each: a dropped term, a wrong sign or index, a transposed
operand.  This checks the pins, not the CUDA path."""
import numpy as np
import pytest

import oracle.attention as orc
from tests import oracle_pins as pins

_real = {name: getattr(orc, name) for name in
         ("_scores", "_apply_mask", "_row_softmax", "_softmax_backward", "visible",
          "forward", "backward", "tiled_forward", "_lse", "window_block_mask", "dilated_block_mask",
          "decode_visible", "decode", "decode_split", "philox4x32_10", "dropout_bytes",
          "forward_dropout", "backward_dropout", "e4m3_decode", "forward_fp8", "fp8_error_model",
          "grad_error_model")}


def _m_no_scale(q, k, scale):
    return q @ k.T


def _m_transposed_scores(q, k, scale):
    s = scale * (q @ k.T)
    return s.T if s.shape[0] == s.shape[1] else s


def _m_mask_zero(s, vis):            # masked entries set to 0 instead of -inf
    return np.where(vis, s, 0.0)


def _m_softmax_no_norm(s):
    p, m, l = _real["_row_softmax"](s)
    return p * l[:, None], m, l


def _m_ds_sign(p, dp, d_row):
    return p * (dp + d_row[:, None])


def _m_ds_no_d(p, dp, d_row):
    return p * dp


def _m_causal_strict(nq, nk, causal=False, block_mask=None, block=128, rows=None):
    vis = _real["visible"](nq, nk, False, block_mask, block, rows)
    if causal:
        r = np.arange(nq) if rows is None else np.asarray(rows)
        vis &= np.arange(nk)[None, :] < np.maximum(r[:, None], 1)
    return vis


def _m_block_transposed(nq, nk, causal=False, block_mask=None, block=128, rows=None):
    bm = None if block_mask is None else np.asarray(block_mask).T
    return _real["visible"](nq, nk, causal, bm, block, rows)


def _m_rows_ignored(nq, nk, causal=False, block_mask=None, block=128, rows=None):
    vis = _real["visible"](nq, nk, causal, block_mask, block, None)
    return vis if rows is None else vis[: len(rows)]


def _m_fwd_kv_swapped(q, k, v, scale, **kw):
    if k.shape == v.shape:
        return _real["forward"](q, v, k, scale, **kw)
    return _real["forward"](q, k, v, scale, **kw)


def _m_bwd_dk_unscaled(q, k, v, do, scale, **kw):
    dq, dk, dv, dvec = _real["backward"](q, k, v, do, scale, **kw)
    return dq, dk / scale, dv, dvec


def _m_bwd_dq_transposed(q, k, v, do, scale, causal=False, block_mask=None, block=128):
    dq, dk, dv, dvec = _real["backward"](q, k, v, do, scale, causal=causal,
                                         block_mask=block_mask, block=block)
    q64, k64, v64, do64 = (np.asarray(x, np.float64) for x in (q, k, v, do))
    for b in range(q64.shape[0]):
        for h in range(q64.shape[1]):
            p, _ = orc.head_probs(q64[b, h], k64[b, h], scale, causal, block_mask, block)
            dp = do64[b, h] @ v64[b, h].T
            ds = p * (dp - (p * dp).sum(1)[:, None])
            dq[b, h] = scale * (ds.T @ k64[b, h])
    return dq, dk, dv, dvec


def _m_tiled_l_no_alpha(q, k, v, scale, Br, Bc, causal=False, block_mask=None, block=128,
                        trace=False):
    """The tiled recurrence with the exp(m - m_new) factor dropped from the l update."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    B, H, N, _ = q.shape
    o_all = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse_all = np.zeros((B, H, N))
    traces = []
    for b in range(B):
        for h in range(H):
            for i0 in range(0, N, Br):
                rows = np.arange(i0, min(N, i0 + Br))
                m = np.full(rows.size, -np.inf)
                l = np.zeros(rows.size)
                o = np.zeros((rows.size, v.shape[-1]))
                tr = []
                for j0 in range(0, k.shape[2], Bc):
                    cols = np.arange(j0, min(k.shape[2], j0 + Bc))
                    s = scale * (q[b, h, rows] @ k[b, h, cols].T)
                    vis = orc.visible(N, k.shape[2], causal, block_mask, block, rows)[:, cols]
                    s = np.where(vis, s, -np.inf)
                    m_new = np.maximum(m, s.max(axis=1))
                    mn = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.exp(np.where(np.isfinite(m), m, -np.inf) - mn)
                    pt = np.exp(s - mn[:, None])
                    l_new = l + pt.sum(axis=1)                       # planted mistake
                    o = ((l * alpha)[:, None] * o + pt @ v[b, h, cols]) / np.where(l_new > 0, l_new, 1)[:, None]
                    m, l = m_new, l_new
                    tr.append((m.copy(), l.copy(), o.copy()))
                o_all[b, h, rows] = o
                lse_all[b, h, rows] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1)), -np.inf)
                traces.append(tr)
    return (o_all, lse_all, traces) if trace else (o_all, lse_all)


def _m_lse_log2(m, l):
    return np.where(l > 0, m + np.log2(np.where(l > 0, l, 1.0)), -np.inf)


def _m_window_right_short(N, left, right, block=128):
    m = _real["window_block_mask"](N, left, right, block)
    nb = m.shape[0]
    for i in range(nb):
        if right > 0 and i + right < nb:
            m[i, i + right] = 0                      # the window stops one block early
    return m


def _m_window_swapped(N, left, right, block=128):
    return _real["window_block_mask"](N, right, left, block)


def _m_dilated_no_dilation(N, window, dilation, causal=False, block=128):
    return _real["dilated_block_mask"](N, window, 1, causal, block)


def _m_dilated_causal_flipped(N, window, dilation, causal=False, block=128):
    m = _real["dilated_block_mask"](N, window, dilation, False, block)
    return np.triu(m) if causal else m


def _m_decode_top_left(nq, L, causal=False):
    vis = np.ones((nq, L), dtype=bool)
    if causal:
        vis &= np.arange(L)[None, :] <= np.arange(nq)[:, None]     # query i at position i
    return vis


def _m_decode_strict(nq, L, causal=False):
    vis = _real["decode_visible"](nq, L, causal)
    if causal:
        pos = L - nq + np.arange(nq)
        vis &= np.arange(L)[None, :] < np.maximum(pos[:, None], 1)
    return vis


def _m_decode_no_seqlens(q, k, v, scale, seqlens=None, causal=False):
    return _real["decode"](q, k, v, scale, None, causal)


def _m_split_unweighted(q, k, v, scale, chunk, seqlens=None, causal=False):
    """Split-KV merge that averages the chunks' outputs with equal weights."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    o, lse = _real["decode_split"](q, k, v, scale, chunk, seqlens, causal)
    B, H, nq, _ = q.shape
    for b in range(B):
        L = k.shape[2] if seqlens is None else int(seqlens[b])
        for h in range(H):
            outs = []
            for c0 in range(0, L, chunk):
                cols = np.arange(c0, min(L, c0 + chunk))
                oc, _ = _real["decode"](q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1, cols], v[b:b + 1, h:h + 1, cols],
                                        scale)
                outs.append(oc[0, 0])
            if len(outs) > 1:
                o[b, h] = np.mean(outs, axis=0)
    return o, lse


def _m_philox_no_bump(ctr, key):
    """Philox with the key held fixed across rounds."""
    c = np.array(ctr, dtype=np.uint64) & 0xFFFFFFFF
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    mask = np.uint64(0xFFFFFFFF)
    for _ in range(10):
        p0 = c[..., 0] * np.uint64(0xD2511F53)
        p1 = c[..., 2] * np.uint64(0xCD9E8D57)
        c = np.stack([(p1 >> np.uint64(32)) ^ c[..., 1] ^ np.uint64(k0), p1 & mask,
                      (p0 >> np.uint64(32)) ^ c[..., 3] ^ np.uint64(k1), p0 & mask], axis=-1)
    return c.astype(np.uint32)


def _m_dropout_transposed(b, h, rows, cols, seed):
    return _real["dropout_bytes"](b, h, cols, rows, seed).T


def _m_dropout_unscaled(q, k, v, scale, p, seed, causal=False, block_mask=None, block=128, b0=0, h0=0):
    o, lse = _real["forward_dropout"](q, k, v, scale, p, seed, causal, block_mask, block, b0, h0)
    return o * (256 - orc.dropout_threshold(p)) / 256.0, lse


def _m_dropout_bwd_no_mask_in_dp(q, k, v, do, scale, p, seed, causal=False, block_mask=None, block=128, b0=0,
                                 h0=0):
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    B, H, N, _ = q.shape
    c = 256.0 / (256 - orc.dropout_threshold(p))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dvec = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            pr, _ = orc.head_probs(q[b, h], k[b, h], scale, causal, block_mask, block)
            zc = orc.dropout_keep(b0 + b, h0 + h, np.arange(N), np.arange(k.shape[2]), p, seed) * c
            dv[b, h] = (pr * zc).T @ do[b, h]
            dp = do[b, h] @ v[b, h].T                       # planted mistake: mask not applied
            d_row = (pr * dp).sum(axis=1)
            ds = pr * (dp - d_row[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
            dvec[b, h] = d_row
    return dq, dk, dv, dvec


def _m_e4m3_bias8(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -7, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 8.0))
    return sign * np.where((c & 0x7F) == 0x7F, np.nan, val)


def _m_e4m3_no_subnormal(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, (c & 0x7).astype(np.float64)
    val = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    return sign * np.where((c & 0x7F) == 0x7F, np.nan, val)


def _m_fp8_v_descale_dropped(q8, k8, v8, qd, kd, vd, scale, causal=False):
    return _real["forward_fp8"](q8, k8, v8, qd, kd, np.ones_like(np.asarray(vd)), scale, causal)


def _m_fp8_sigma_halved(o, probs, v, rel=2.0 ** -4):
    bound, sigma = _real["fp8_error_model"](o, probs, v, rel)
    return bound, sigma / 2


def _m_grad_sigma_halved(*a, **kw):
    sig, acc = _real["grad_error_model"](*a, **kw)
    return tuple(x / 2 for x in sig), acc


def _m_grad_ds_rounding_dropped(q, k, v, do, scale, causal=False, block_mask=None, block=128, row_chunk=1024,
                                u=orc.BF16_U, f32=orc.FP32_STEP):
    """The model without the bf16 rounding of dS and O (dQ and dK keep only fp32 terms)."""
    sig, acc = _real["grad_error_model"](q, k, v, do, scale, causal, block_mask, block, row_chunk, u=0.0, f32=f32)
    sig_v, _ = _real["grad_error_model"](q, k, v, do, scale, causal, block_mask, block, row_chunk, u=u, f32=f32)
    return (sig[0], sig[1], sig_v[2]), acc


MUTANTS = {
    "scale_dropped": ("_scores", _m_no_scale),
    "scores_transposed": ("_scores", _m_transposed_scores),
    "mask_as_zero": ("_apply_mask", _m_mask_zero),
    "softmax_unnormalised": ("_row_softmax", _m_softmax_no_norm),
    "dS_sign_flipped": ("_softmax_backward", _m_ds_sign),
    "dS_missing_D": ("_softmax_backward", _m_ds_no_d),
    "causal_off_by_one": ("visible", _m_causal_strict),
    "block_mask_transposed": ("visible", _m_block_transposed),
    "visible_rows_ignored": ("visible", _m_rows_ignored),
    "forward_kv_swapped": ("forward", _m_fwd_kv_swapped),
    "dK_scale_dropped": ("backward", _m_bwd_dk_unscaled),
    "dQ_dS_transposed": ("backward", _m_bwd_dq_transposed),
    "tiled_l_rescale_dropped": ("tiled_forward", _m_tiled_l_no_alpha),
    "lse_wrong_base": ("_lse", _m_lse_log2),
    "window_right_short": ("window_block_mask", _m_window_right_short),
    "window_sides_swapped": ("window_block_mask", _m_window_swapped),
    "dilated_without_dilation": ("dilated_block_mask", _m_dilated_no_dilation),
    "dilated_causal_flipped": ("dilated_block_mask", _m_dilated_causal_flipped),
    "decode_causal_top_left": ("decode_visible", _m_decode_top_left),
    "decode_causal_strict": ("decode_visible", _m_decode_strict),
    "decode_ignores_seqlens": ("decode", _m_decode_no_seqlens),
    "decode_split_unweighted": ("decode_split", _m_split_unweighted),
    "philox_key_not_advanced": ("philox4x32_10", _m_philox_no_bump),
    "dropout_mask_transposed": ("dropout_bytes", _m_dropout_transposed),
    "dropout_output_unscaled": ("forward_dropout", _m_dropout_unscaled),
    "dropout_grad_mask_missing": ("backward_dropout", _m_dropout_bwd_no_mask_in_dp),
    "e4m3_exponent_bias_8": ("e4m3_decode", _m_e4m3_bias8),
    "e4m3_subnormals_as_normal": ("e4m3_decode", _m_e4m3_no_subnormal),
    "fp8_v_descale_dropped": ("forward_fp8", _m_fp8_v_descale_dropped),
    "fp8_sigma_halved": ("fp8_error_model", _m_fp8_sigma_halved),
    "grad_sigma_halved": ("grad_error_model", _m_grad_sigma_halved),
    "grad_ds_rounding_dropped": ("grad_error_model", _m_grad_ds_rounding_dropped),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(orc, attr, fn)
    failures = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, IndexError):
            failures.append(pin.__name__)
    assert failures, f"mutant {name} passed every pin"
