"""Plain, slow, fp64 statement of what the fused LM-head cross-entropy computes.

TEST INFRASTRUCTURE: only tests, the smoke check and the benchmark's CPU
baseline may use this module. It shares no code with the CUDA library.

Notation (Trillion Labs note, "Cross Entropy를 다시 보면"; PyTorch 2.13
LinearCrossEntropyLoss chapter, "먼저 수식에서 없앨 수 있는 tensor를 찾는다"):
H [N,D] hidden rows, W [V,D] LM-head weight, y [N] targets with
ignore_index = -100.

    z_n     = H_n W^T                              (one logit row)
    LSE_n   = m_n + log sum_v exp(z_nv - m_n),      m_n = max_v z_nv
    loss    = sum_{valid n} (LSE_n - z_{n,y_n}) / count    (0 when count = 0)
    dZ_nv   = (g / count) * valid_n * (exp(z_nv - LSE_n) - [v = y_n])
    dH      = dZ W,   dW = dZ^T H

The stable max-shifted LSE is the one Cut Cross-Entropy prescribes
("Cut Your Losses in Large-Vocabulary Language Models", Sec. 4.2, Alg. 2);
the softmax in the backward is exp(z - LSE) with no renormalisation (Sec. 4.3).
The loss is the negative of that paper's Eq. 4 log-likelihood, averaged over
non-ignored rows with the count clamped to at least one (the note's chunked
cross-entropy listing divides by count.clamp_min(1)), so dZ is
softmax - onehot (the note's and the chapter's gradient formula) rather than
the paper's onehot - softmax (Alg. 4).

All arithmetic is fp64 on exactly widened bf16 inputs; matrix products use the
library matmul. Rows are processed in blocks only to bound memory: every
output element is still one plain sum.
"""

from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100
_BLOCK_BYTES = 256 << 20


def inputs_f64(h_bits: np.ndarray, w_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Widen bf16 bit patterns (uint16) to fp64 exactly."""
    def widen(b):
        return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
            np.float32).astype(np.float64)
    return widen(h_bits), widen(w_bits)


def _row_blocks(n: int, vocab: int):
    step = max(1, _BLOCK_BYTES // max(1, vocab * 8))
    for r0 in range(0, n, step):
        yield r0, min(n, r0 + step)


def logits(H: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z = H W^T in fp64 (the LM-head projection)."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """Per-row log-sum-exp, shifted by the row maximum for stability."""
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def valid_count(y: np.ndarray, ignore_index: int = IGNORE_INDEX) -> int:
    return int(np.count_nonzero(np.asarray(y) != ignore_index))


def _check_targets(y, vocab, ignore_index):
    y = np.asarray(y, dtype=np.int64)
    bad = (y != ignore_index) & ((y < 0) | (y >= vocab))
    if np.any(bad):
        raise ValueError("target outside [0, V) that is not ignore_index")
    return y


def lse_rows(H: np.ndarray, W: np.ndarray, rows) -> np.ndarray:
    """LSE_n for the listed rows only (each needs just H_n and all of W)."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.float64)
    for r0, r1 in _row_blocks(rows.shape[0], W.shape[0]):
        out[r0:r1] = logsumexp_rows(logits(H[rows[r0:r1]], W))
    return out


def forward(H: np.ndarray, W: np.ndarray, y: np.ndarray, ignore_index: int = IGNORE_INDEX):
    """Per-row LSE, mean loss over valid rows and the valid count."""
    n, vocab = H.shape[0], W.shape[0]
    y = _check_targets(y, vocab, ignore_index)
    lse = np.empty(n, dtype=np.float64)
    total = 0.0
    for r0, r1 in _row_blocks(n, vocab):
        z = logits(H[r0:r1], W)
        lse[r0:r1] = logsumexp_rows(z)
        for i in range(r1 - r0):
            t = y[r0 + i]
            if t != ignore_index:
                total += lse[r0 + i] - z[i, t]
    count = valid_count(y, ignore_index)
    loss = total / max(count, 1)
    return lse, loss, count


def loss_value(H, W, y, ignore_index: int = IGNORE_INDEX) -> float:
    return forward(H, W, y, ignore_index)[1]


def _dlogits_block(z, lse_blk, y_blk, scale, ignore_index):
    dz = np.exp(z - lse_blk[:, None])
    for i in range(z.shape[0]):
        t = y_blk[i]
        if t == ignore_index:
            dz[i, :] = 0.0
        else:
            dz[i, t] -= 1.0
    return dz * scale


def dlogits(H, W, y, grad_loss: float = 1.0, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """The full dZ [N,V] (small inputs only: this is the array the method avoids)."""
    y = _check_targets(y, W.shape[0], ignore_index)
    z = logits(H, W)
    lse = logsumexp_rows(z)
    scale = grad_loss / max(valid_count(y, ignore_index), 1)
    return _dlogits_block(z, lse, y, scale, ignore_index)


def forward_backward(H, W, y, grad_loss: float = 1.0, ignore_index: int = IGNORE_INDEX):
    """LSE [N], loss, dH [N,D], dW [V,D], count; no [N,V] array beyond a row block."""
    n, vocab = H.shape[0], W.shape[0]
    y = _check_targets(y, vocab, ignore_index)
    count = valid_count(y, ignore_index)
    scale = grad_loss / max(count, 1)
    lse = np.empty(n, dtype=np.float64)
    dH = np.zeros(H.shape, dtype=np.float64)
    dW = np.zeros(W.shape, dtype=np.float64)
    total = 0.0
    for r0, r1 in _row_blocks(n, vocab):
        z = logits(H[r0:r1], W)
        lse[r0:r1] = logsumexp_rows(z)
        for i in range(r1 - r0):
            t = y[r0 + i]
            if t != ignore_index:
                total += lse[r0 + i] - z[i, t]
        dz = _dlogits_block(z, lse[r0:r1], y[r0:r1], scale, ignore_index)
        dH[r0:r1] = dz @ W
        dW += dz.T @ H[r0:r1]
    loss = total / max(count, 1)
    return lse, loss, dH, dW, count


def dH_rows(H, W, y, rows, grad_loss: float = 1.0, ignore_index: int = IGNORE_INDEX):
    """dH_n for the listed rows: needs LSE_n, the global valid count and W."""
    y = _check_targets(y, W.shape[0], ignore_index)
    rows = np.asarray(rows, dtype=np.int64)
    scale = grad_loss / max(valid_count(y, ignore_index), 1)
    out = np.empty((rows.shape[0], W.shape[1]), dtype=np.float64)
    for r0, r1 in _row_blocks(rows.shape[0], W.shape[0]):
        sel = rows[r0:r1]
        z = logits(H[sel], W)
        dz = _dlogits_block(z, logsumexp_rows(z), y[sel], scale, ignore_index)
        out[r0:r1] = dz @ W
    return out


def dW_rows(H, W, y, lse, vocab_ids, grad_loss: float = 1.0, ignore_index: int = IGNORE_INDEX):
    """dW_v for the listed vocabulary rows, given the oracle's own LSE of all rows.

    dW_v = (g / count) sum_{valid n} (exp(z_nv - LSE_n) - [y_n = v]) H_n.
    """
    y = _check_targets(y, W.shape[0], ignore_index)
    vocab_ids = np.asarray(vocab_ids, dtype=np.int64)
    scale = grad_loss / max(valid_count(y, ignore_index), 1)
    zc = logits(H, W[vocab_ids])                       # [N, k]
    p = np.exp(zc - np.asarray(lse, dtype=np.float64)[:, None])
    valid = y != ignore_index
    p[~valid, :] = 0.0
    for j, v in enumerate(vocab_ids):
        p[valid & (y == v), j] -= 1.0
    return scale * (p.T @ H)


def average_logits(H, W, y, bias=None, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """Average logit of every vocabulary entry over the valid rows.

    Cut Cross-Entropy, Sec. 4.3 "Vocabulary sorting": the forward pass
    accumulates, per token, its logit averaged over the batch, and the
    backward groups the vocabulary by that average. Read here as
    a_v = sum_{valid n} z_nv / count, with z_nv = H_n W_v^T (+ b_v); ignored
    rows carry no gradient, so they take no part; all zero when count = 0.
    Computed from the logits themselves, a row block at a time.
    """
    n, vocab = H.shape[0], W.shape[0]
    y = _check_targets(y, vocab, ignore_index)
    valid = y != ignore_index
    count = int(valid.sum())
    total = np.zeros(vocab, dtype=np.float64)
    for r0, r1 in _row_blocks(n, vocab):
        z = logits(H[r0:r1], W)
        if bias is not None:
            z = z + np.asarray(bias, dtype=np.float64)[None, :]
        total += z[valid[r0:r1]].sum(axis=0)
    return total / count if count > 0 else total


def vocabulary_order(avg: np.ndarray) -> np.ndarray:
    """Vocabulary ids by decreasing average logit, equal averages in id order.

    order[i] is the id placed at sorted position i; the backward then cuts
    the sorted vocabulary into blocks, so ids of similar average logit share
    a block (Cut Cross-Entropy, Sec. 4.3 "Vocabulary sorting").
    """
    return np.argsort(-np.asarray(avg, dtype=np.float64), kind="stable")


def forward_backward_filtered(H, W, y, eps: float, tile_rows: int, tile_cols: int,
                              grad_loss: float = 1.0, ignore_index: int = IGNORE_INDEX,
                              filter_dH: bool = True, filter_dW: bool = True, dH_tile_rows: int | None = None,
                              vocab_order=None):
    """Gradient filtering of Cut Cross-Entropy Alg. 4, emulated in fp64.

    The dZ matrix is cut into tile_rows x tile_cols tiles aligned at 0; a tile
    whose unscaled gradient G = softmax - onehot has every |G| < eps (ignored
    rows count as G = 0) contributes nothing to dH or dW. filter_dH /
    filter_dW = False computes that gradient from the full G (the paper's
    CCE-FullE / CCE-FullC variants). dH_tile_rows (a multiple of tile_rows,
    default tile_rows) gives dH its own, taller mask: a tile_rows-high tile
    then drops out of dH only when its whole dH_tile_rows-high block does.
    vocab_order (a permutation of the ids, e.g. vocabulary_order's) lays the
    columns out in that order before the tiles are cut, so column block j
    holds ids vocab_order[j*tile_cols : (j+1)*tile_cols] (Sec. 4.3,
    "Vocabulary sorting"); dW is returned in id order.
    Returns the same tuple as forward_backward plus the fraction of
    tile_rows x tile_cols tiles skipped.
    """
    n, vocab = H.shape[0], W.shape[0]
    y = _check_targets(y, vocab, ignore_index)
    if vocab_order is not None:
        order = np.asarray(vocab_order, dtype=np.int64)
        if order.shape != (vocab,) or not np.array_equal(np.sort(order), np.arange(vocab)):
            raise ValueError("vocab_order must be a permutation of the vocabulary ids")
        position = np.empty(vocab, dtype=np.int64)
        position[order] = np.arange(vocab)
        y_sorted = np.where(y == ignore_index, y, position[np.where(y == ignore_index, 0, y)])
        if ignore_index >= 0:
            # keep ignored rows ignored even where a position equals ignore_index
            y_sorted = np.where(y == ignore_index, -1, y_sorted)
            ignore_sorted = -1
        else:
            ignore_sorted = ignore_index
        lse, loss, dH, dW_sorted, count, frac = forward_backward_filtered(
            H, W[order], y_sorted, eps, tile_rows, tile_cols, grad_loss, ignore_sorted, filter_dH, filter_dW,
            dH_tile_rows)
        dW = np.empty_like(dW_sorted)
        dW[order] = dW_sorted
        return lse, loss, dH, dW, count, frac
    count = valid_count(y, ignore_index)
    scale = grad_loss / max(count, 1)
    lse, loss, _ = forward(H, W, y, ignore_index)
    dH = np.zeros(H.shape, dtype=np.float64)
    dW = np.zeros(W.shape, dtype=np.float64)
    tiles = skipped = 0
    hr = tile_rows if dH_tile_rows is None else dH_tile_rows
    if hr % tile_rows != 0:
        raise ValueError("dH_tile_rows must be a multiple of tile_rows")
    for b0 in range(0, n, hr):
        b1 = min(n, b0 + hr)
        z = logits(H[b0:b1], W)
        g_full = _dlogits_block(z, lse[b0:b1], y[b0:b1], 1.0, ignore_index)
        g_w = g_full.copy()                      # dW mask: tile_rows x tile_cols
        g_h = g_full.copy()                      # dH mask: hr x tile_cols
        for c0 in range(0, vocab, tile_cols):
            c1 = min(vocab, c0 + tile_cols)
            small = []
            for r0 in range(0, b1 - b0, tile_rows):
                r1 = min(b1 - b0, r0 + tile_rows)
                tiles += 1
                s_ = bool(np.all(np.abs(g_full[r0:r1, c0:c1]) < eps))
                small.append(s_)
                if s_:
                    skipped += 1
                    g_w[r0:r1, c0:c1] = 0.0
            if all(small):
                g_h[:, c0:c1] = 0.0
        dH[b0:b1] = ((g_h if filter_dH else g_full) * scale) @ W
        dW += ((g_w if filter_dW else g_full) * scale).T @ H[b0:b1]
    return lse, loss, dH, dW, count, skipped / max(tiles, 1)


def forward_backward_ex(H, W, y, bias=None, reduction: str = "mean", grad=1.0,
                        ignore_index: int = IGNORE_INDEX, need_grad: bool = True):
    """The general form: optional bias, reduction mean | sum | none.

    With a bias b [V] the logits are z_n = H_n W^T + b (the PyTorch 2.13
    chapter's linear_bias argument of F.linear_cross_entropy). Per-row losses
    l_n = LSE_n - z_{n,y_n} (0 on ignored rows) are reduced to
      mean: sum_n l_n / max(count, 1),  sum: sum_n l_n,  none: the vector l.
    `grad` is the upstream gradient of the result: a scalar for mean/sum, a
    length-N vector for none. dZ_nv = s_n * valid_n * (exp(z_nv - LSE_n) - [v = y_n])
    with s_n = grad/max(count,1), grad, or grad[n]; dH = dZ W, dW = dZ^T H,
    db = sum_n dZ_n. Returns a dict with lse, loss, count and, if need_grad,
    dH, dW, db (db is None without a bias).
    """
    n, vocab = H.shape[0], W.shape[0]
    y = _check_targets(y, vocab, ignore_index)
    if reduction not in ("mean", "sum", "none"):
        raise ValueError(reduction)
    count = valid_count(y, ignore_index)
    valid = y != ignore_index
    if reduction == "none":
        g = np.broadcast_to(np.asarray(grad, dtype=np.float64), (n,))
        row_scale = g
    else:
        g0 = float(grad)
        row_scale = np.full(n, g0 / max(count, 1) if reduction == "mean" else g0)
    lse = np.empty(n, dtype=np.float64)
    rows_loss = np.zeros(n, dtype=np.float64)
    dH = np.zeros(H.shape, dtype=np.float64) if need_grad else None
    dW = np.zeros(W.shape, dtype=np.float64) if need_grad else None
    db = np.zeros(vocab, dtype=np.float64) if (need_grad and bias is not None) else None
    b = None if bias is None else np.asarray(bias, dtype=np.float64)
    for r0, r1 in _row_blocks(n, vocab):
        z = logits(H[r0:r1], W)
        if b is not None:
            z = z + b[None, :]
        lse[r0:r1] = logsumexp_rows(z)
        for i in range(r1 - r0):
            if valid[r0 + i]:
                rows_loss[r0 + i] = lse[r0 + i] - z[i, y[r0 + i]]
        if need_grad:
            dz = _dlogits_block(z, lse[r0:r1], y[r0:r1], 1.0, ignore_index) * row_scale[r0:r1, None]
            dH[r0:r1] = dz @ W
            dW += dz.T @ H[r0:r1]
            if db is not None:
                db += dz.sum(axis=0)
    if reduction == "none":
        loss = rows_loss
    elif reduction == "sum":
        loss = float(rows_loss.sum())
    else:
        loss = float(rows_loss.sum()) / max(count, 1)
    return {"lse": lse, "loss": loss, "count": count, "dH": dH, "dW": dW, "db": db}


def adamw_step(param, grad, m, v, step: int, lr: float, beta1: float, beta2: float, eps: float,
               weight_decay: float):
    """One AdamW step, elementwise in fp64; returns the new (param, m, v).

    The optimizer the FORGE explainer fuses into the weight-gradient tiles
    ("FORGE: Fused On-Register Gradient Elimination for Memory-Efficient LLM
    Training", Sec. 2, core mechanism: AdamW named as the example). The page
    prints no formula; this is AdamW with decoupled weight decay as
    Loshchilov and Hutter define it and torch.optim.AdamW computes it:
        param <- param * (1 - lr * weight_decay)
        m <- beta1 m + (1 - beta1) g,   v <- beta2 v + (1 - beta2) g^2
        param <- param - lr * (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
    with t = step >= 1, the step being taken.
    """
    if step < 1:
        raise ValueError("step counts from 1")
    p = np.asarray(param, dtype=np.float64) * (1.0 - lr * weight_decay)
    g = np.asarray(grad, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** step)
    v_hat = v / (1.0 - beta2 ** step)
    p = p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v


def forward_backward_adamw(H, W, y, master, m, v, hparams: dict, grad_loss: float = 1.0,
                           ignore_index: int = IGNORE_INDEX):
    """The LM-head step with W's AdamW update fused into its gradient.

    FORGE applies the optimizer to each weight-gradient tile as soon as the
    tile is complete, so the gradient is never stored; for an elementwise
    optimizer the page states the result equals the usual two-phase step
    (Sec. 2, exactness). The oracle is therefore the two-phase step: dW of
    forward_backward (on the bf16 W the forward used), then adamw_step on
    the fp32 master weights. Returns a dict with lse, loss, count, dH and
    the new master, m and v.
    """
    lse, loss, dH, dW, count = forward_backward(H, W, y, grad_loss=grad_loss, ignore_index=ignore_index)
    p, m2, v2 = adamw_step(master, dW, m, v, **hparams)
    return {"lse": lse, "loss": loss, "count": count, "dH": dH, "dW": dW, "master": p, "m": m2, "v": v2}
