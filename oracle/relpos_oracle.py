"""CPU float64 oracle for global attention with decomposed relative-position bias.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import or call this module.  The
product path (the CUDA library and its binding) never does, and this module
imports nothing from the product.

Source: vLLM PR #55629 page ("为 DeepEncoder 全局注意力融合相对位置偏置到 Triton 内核").

* Section 关键源码片段 (key source excerpt): ``add_decomposed_rel_pos(q,
  rel_pos_h, rel_pos_w, (H, W), (H, W))`` returns ``rel_h`` and ``rel_w``; the
  fallback branch builds ``attn_bias = (rel_h + rel_w).view(B, heads, HW, H*W)``
  and calls ``F.scaled_dot_product_attention(q, k, v, attn_mask=attn_bias)``.
  That additive-mask call *defines* the result:
  ``out = softmax(scale * q k^T + bias) v`` with ``scale = d**-0.5``.
* The page does not print the body of ``add_decomposed_rel_pos``.  Reading
  taken (SAM-style decomposed relative position, consistent with the table
  lengths 2H-1 / 2W-1 and the ``.view`` above):
  ``rel_h[n, kh] = q_n . rel_pos_h[qh(n) - kh + H - 1]`` and
  ``rel_w[n, kw] = q_n . rel_pos_w[qw(n) - kw + W - 1]``, with row-major token
  order ``n = qh*W + qw`` and key order ``m = kh*W + kw``; the projection uses
  the unscaled q (it runs before SDPA applies the scale).
* Section 风险与影响 (risks): the fast path accumulates in fp32; the oracle is
  exact float64 softmax (a row-max shift is used only to avoid overflow).

All functions take array-likes (converted to float64) shaped
``q, k, v: [BH, N, d]``, ``rel_pos_h: [2H-1, d]``, ``rel_pos_w: [2W-1, d]``,
``rel_h: [BH, N, H]``, ``rel_w: [BH, N, W]``.

Backward (training use; the pages print no backward).  Reading taken: the
gradient of the definition above, by the chain rule.  With
``Z = scale * q k^T + Bias``, ``P = softmax_rows(Z)``, ``O = P v`` and an
upstream gradient ``dO``:
``dv = P^T dO``; ``dP = dO v^T``; ``dZ = P * (dP - D)`` with
``D[n] = sum_m P[n, m] dP[n, m] = dO[n] . O[n]``; ``dq = scale dZ k``;
``dk = scale dZ^T q``; the bias gradient is ``dZ`` itself, so
``drel_h[n, kh] = sum_kw dZ[n, kh*W + kw]`` and
``drel_w[n, kw] = sum_kh dZ[n, kh*W + kw]``; through the projection,
``dq[n] += sum_kh drel_h[n, kh] rel_pos_h[qh - kh + H - 1]`` (and the same for
w), and ``drel_pos_h[i] = sum over (b, n, kh) with qh - kh + H - 1 = i of
drel_h[b, n, kh] q[b, n]`` (tables are shared by every batch and head).

Pins: every function here is pinned in ``tests/test_oracle.py`` against
brute force, the library SDPA routine, closed forms, central finite
differences (the backward) and hand-derived golden fixtures; none is
"parity unpinned".
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def rel_index(length: int) -> np.ndarray:
    """Table row used for query coordinate a and key coordinate b: ``a - b + length - 1``."""
    a = np.arange(length)[:, None]
    b = np.arange(length)[None, :]
    return a - b + length - 1


def project(q, rel_pos_h, rel_pos_w, H: int, W: int):
    """Decomposed rel-pos projection: ``(rel_h [BH,N,H], rel_w [BH,N,W])`` in float64."""
    q = _f64(q)
    th, tw = _f64(rel_pos_h), _f64(rel_pos_w)
    BH, N, d = q.shape
    if N != H * W:
        raise ValueError("N must equal H*W")
    if th.shape != (2 * H - 1, d) or tw.shape != (2 * W - 1, d):
        raise ValueError("tables must be [2H-1, d] and [2W-1, d]")
    qg = q.reshape(BH, H, W, d)                 # token n = qh*W + qw
    Rh = th[rel_index(H)]                       # [qh, kh, d]
    Rw = tw[rel_index(W)]                       # [qw, kw, d]
    rel_h = np.einsum("bhwc,hkc->bhwk", qg, Rh, optimize=True).reshape(BH, N, H)
    rel_w = np.einsum("bhwc,wkc->bhwk", qg, Rw, optimize=True).reshape(BH, N, W)
    return rel_h, rel_w


def project_rows(q_rows, rows, rel_pos_h, rel_pos_w, H: int, W: int):
    """Projection for selected token rows only: ``q_rows [R, d]``, token indices ``rows [R]``."""
    q_rows = _f64(q_rows)
    rows = np.asarray(rows, dtype=np.int64)
    th, tw = _f64(rel_pos_h), _f64(rel_pos_w)
    qh, qw = rows // W, rows % W
    Rh = th[qh[:, None] - np.arange(H)[None, :] + H - 1]      # [R, H, d]
    Rw = tw[qw[:, None] - np.arange(W)[None, :] + W - 1]      # [R, W, d]
    return np.einsum("rc,rkc->rk", q_rows, Rh), np.einsum("rc,rkc->rk", q_rows, Rw)


def dense_bias(rel_h_b, rel_w_b, H: int, W: int) -> np.ndarray:
    """The materialised bias of one (batch, head): ``Bias[n, kh*W + kw] = rel_h[n, kh] + rel_w[n, kw]``."""
    rel_h_b, rel_w_b = _f64(rel_h_b), _f64(rel_w_b)
    R = rel_h_b.shape[0]
    return (rel_h_b[:, :, None] + rel_w_b[:, None, :]).reshape(R, H * W)


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    z = logits - logits.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def attention(q, k, v, rel_h, rel_w, H: int, W: int, scale: float) -> np.ndarray:
    """``out[b] = softmax(scale * q[b] k[b]^T + Bias[b]) v[b]`` for every (batch, head) b."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    rel_h, rel_w = _f64(rel_h), _f64(rel_w)
    BH, N, _ = q.shape
    if N != H * W:
        raise ValueError("N must equal H*W")
    out = np.empty((BH, N, v.shape[2]), dtype=np.float64)
    for b in range(BH):
        logits = scale * (q[b] @ k[b].T) + dense_bias(rel_h[b], rel_w[b], H, W)
        out[b] = _softmax_rows(logits) @ v[b]
    return out


def attention_rows(q, k, v, rel_h_rows, rel_w_rows, b: int, rows, H: int, W: int, scale: float) -> np.ndarray:
    """Output rows ``rows`` of head ``b`` only; ``rel_*_rows`` hold the bias of those rows."""
    rows = np.asarray(rows, dtype=np.int64)
    qb = _f64(q[b])[rows]
    kb, vb = _f64(k[b]), _f64(v[b])
    logits = scale * (qb @ kb.T) + dense_bias(rel_h_rows, rel_w_rows, H, W)
    return _softmax_rows(logits) @ vb


def fused(q, k, v, rel_pos_h, rel_pos_w, H: int, W: int, scale: float) -> np.ndarray:
    """Projection followed by attention, the whole path in float64."""
    rel_h, rel_w = project(q, rel_pos_h, rel_pos_w, H, W)
    return attention(q, k, v, rel_h, rel_w, H, W, scale)


def fused_rows(q, k, v, rel_pos_h, rel_pos_w, b: int, rows, H: int, W: int, scale: float) -> np.ndarray:
    """Selected output rows of head ``b`` of :func:`fused`."""
    rows = np.asarray(rows, dtype=np.int64)
    rh, rw = project_rows(_f64(q[b])[rows], rows, rel_pos_h, rel_pos_w, H, W)
    return attention_rows(q, k, v, rh, rw, b, rows, H, W, scale)


def lse2(q, k, rel_h, rel_w, H: int, W: int, scale: float) -> np.ndarray:
    """Base-2 log-sum-exp of every row's logits: ``log2 sum_m exp(Z[n, m])``, shape ``[BH, N]``."""
    q, k = _f64(q), _f64(k)
    BH, N, _ = q.shape
    out = np.empty((BH, N), dtype=np.float64)
    for b in range(BH):
        z = scale * (q[b] @ k[b].T) + dense_bias(_f64(rel_h[b]), _f64(rel_w[b]), H, W)
        mx = z.max(axis=-1)
        out[b] = (mx + np.log(np.exp(z - mx[:, None]).sum(axis=-1))) / np.log(2.0)
    return out


def attention_backward(q, k, v, rel_h, rel_w, H: int, W: int, scale: float, dout):
    """Gradients of ``sum(dout * attention(...))``: ``(dq, dk, dv, drel_h, drel_w)`` in float64."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    rel_h, rel_w = _f64(rel_h), _f64(rel_w)
    BH, N, _ = q.shape
    if N != H * W:
        raise ValueError("N must equal H*W")
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    drel_h, drel_w = np.zeros_like(rel_h), np.zeros_like(rel_w)
    for b in range(BH):
        z = scale * (q[b] @ k[b].T) + dense_bias(rel_h[b], rel_w[b], H, W)
        p = _softmax_rows(z)
        o = p @ v[b]
        dv[b] = p.T @ dout[b]
        dp = dout[b] @ v[b].T
        d = (dout[b] * o).sum(axis=-1)
        dz = p * (dp - d[:, None])
        dq[b] = scale * (dz @ k[b])
        dk[b] = scale * (dz.T @ q[b])
        dz3 = dz.reshape(N, H, W)                # key m = kh*W + kw
        drel_h[b] = dz3.sum(axis=2)
        drel_w[b] = dz3.sum(axis=1)
    return dq, dk, dv, drel_h, drel_w


def fused_backward(q, k, v, rel_pos_h, rel_pos_w, H: int, W: int, scale: float, dout):
    """Gradients of ``sum(dout * fused(...))``: ``(dq, dk, dv, drel_pos_h, drel_pos_w)`` in float64."""
    q = _f64(q)
    th, tw = _f64(rel_pos_h), _f64(rel_pos_w)
    BH, N, d = q.shape
    rel_h, rel_w = project(q, th, tw, H, W)
    dq, dk, dv, drel_h, drel_w = attention_backward(q, k, v, rel_h, rel_w, H, W, scale, dout)
    qg = q.reshape(BH, H, W, d)
    gh = drel_h.reshape(BH, H, W, H)             # [b, qh, qw, kh]
    gw = drel_w.reshape(BH, H, W, W)             # [b, qh, qw, kw]
    Rh = th[rel_index(H)]                        # [qh, kh, d]
    Rw = tw[rel_index(W)]                        # [qw, kw, d]
    dq = dq + (np.einsum("bhwk,hkc->bhwc", gh, Rh, optimize=True)
               + np.einsum("bhwk,wkc->bhwc", gw, Rw, optimize=True)).reshape(BH, N, d)
    dth, dtw = np.zeros_like(th), np.zeros_like(tw)
    # scatter-add: table row rel_index[qh, kh] receives sum_b sum_qw drel_h[b, qh, qw, kh] q[b, qh, qw]
    ch = np.einsum("bhwk,bhwc->hkc", gh, qg, optimize=True)      # [qh, kh, d]
    cw = np.einsum("bhwk,bhwc->wkc", gw, qg, optimize=True)      # [qw, kw, d]
    np.add.at(dth, rel_index(H).reshape(-1), ch.reshape(-1, d))
    np.add.at(dtw, rel_index(W).reshape(-1), cw.reshape(-1, d))
    return dq, dk, dv, dth, dtw
