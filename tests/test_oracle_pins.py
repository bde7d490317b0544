"""Pins for the fp64 oracle: closed forms, invariants, a library cross-check,
finite differences and symmetries. None of these re-uses the oracle's code.

The facts pinned come from the pages: the loss is logsumexp(z) - z_y with
z = h W^T and gradient softmax - onehot (Trillion Labs note, "Cross Entropy를
다시 보면"); the mean is over non-ignored rows with the count clamped to one
(the note's chunked cross-entropy listing); dH = dZ W and dW = dZ^T H
(PyTorch 2.13 LinearCrossEntropyLoss chapter, "먼저 수식에서 없앨 수 있는 tensor를
찾는다"); softmax = exp(z - LSE) (Cut Cross-Entropy, Sec. 4.3).
"""

import math

import numpy as np
import pytest
import torch

import oracle

IGN = -100


def _rand(seed, n, d, v, w_scale=0.5, ignore=()):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((n, d))
    W = rng.standard_normal((v, d)) * w_scale
    y = rng.integers(0, v, size=n).astype(np.int64)
    for i in ignore:
        y[i] = IGN
    return H, W, y


def test_w_zero_gives_log_v_and_closed_form_gradients():
    n, d, v = 7, 5, 13
    H, _, y = _rand(1, n, d, v, ignore=(2, 5))
    W = np.zeros((v, d))
    g = 1.7
    lse, loss, dH, dW, count = oracle.forward_backward(H, W, y, grad_loss=g)
    assert count == 5
    assert np.all(np.abs(lse - math.log(v)) < 1e-14)
    assert abs(loss - math.log(v)) < 1e-14
    assert np.all(dH == 0.0)
    # dW_v = (g/count) * sum_{valid n} (1/V - [y_n = v]) H_n, written out by loops.
    expect = np.zeros((v, d))
    for vv in range(v):
        for i in range(n):
            if y[i] == IGN:
                continue
            coef = 1.0 / v - (1.0 if y[i] == vv else 0.0)
            for k in range(d):
                expect[vv, k] += coef * H[i, k]
    expect *= g / count
    assert np.max(np.abs(dW - expect)) < 1e-13


def test_w_zero_headline_vocab_value():
    # log(151552) for the Gravity-16B-A3B vocabulary.
    H = np.ones((2, 8))
    W = np.zeros((151552, 8))
    lse, loss, _ = oracle.forward(H, W, np.array([3, 151551]))
    assert abs(loss - 11.9286841) < 1e-6
    assert abs(lse[0] - math.log(151552)) < 1e-13


def test_dz_rows_sum_to_zero_and_ignored_rows_are_zero():
    H, W, y = _rand(2, 9, 6, 31, w_scale=1.0, ignore=(0, 4))
    g = 3.0
    dz = oracle.dlogits(H, W, y, grad_loss=g)
    count = 7
    for i in range(9):
        if y[i] == IGN:
            assert np.all(dz[i] == 0.0)
        else:
            assert abs(dz[i].sum()) < 1e-14
            assert dz[i, y[i]] < 0
            assert np.all(dz[i] >= -g / count - 1e-15)
            assert np.all(dz[i] <= g / count + 1e-15)


def test_ignored_rows_have_exactly_zero_dh():
    H, W, y = _rand(3, 12, 8, 40, ignore=(1, 7, 11))
    _, _, dH, _, _ = oracle.forward_backward(H, W, y)
    for i in (1, 7, 11):
        assert np.all(dH[i] == 0.0)
    assert np.all(np.abs(dH[0]) > 0)


def test_central_finite_differences():
    n, d, v = 6, 5, 11
    H, W, y = _rand(4, n, d, v, w_scale=1.0, ignore=(3,))
    _, _, dH, dW, _ = oracle.forward_backward(H, W, y)
    h = 1e-6
    for i in range(n):
        for k in range(d):
            Hp, Hm = H.copy(), H.copy()
            Hp[i, k] += h
            Hm[i, k] -= h
            fd = (oracle.loss_value(Hp, W, y) - oracle.loss_value(Hm, W, y)) / (2 * h)
            assert abs(fd - dH[i, k]) <= 1e-6 * max(1.0, abs(dH[i, k])) + 1e-9
    for vv in range(v):
        for k in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[vv, k] += h
            Wm[vv, k] -= h
            fd = (oracle.loss_value(H, Wp, y) - oracle.loss_value(H, Wm, y)) / (2 * h)
            assert abs(fd - dW[vv, k]) <= 1e-6 * max(1.0, abs(dW[vv, k])) + 1e-9


@pytest.mark.parametrize("seed,n,d,v", [(5, 17, 12, 50), (6, 33, 8, 257), (7, 4, 3, 2)])
def test_matches_explicit_full_logits_library_cross_entropy(seed, n, d, v):
    H, W, y = _rand(seed, n, d, v, w_scale=2.0, ignore=(0,) if n > 1 else ())
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    z = Ht @ Wt.T
    ref = torch.nn.functional.cross_entropy(z, torch.tensor(y), ignore_index=IGN, reduction="mean")
    ref.backward()
    lse_ref = torch.logsumexp(z.detach(), dim=1).numpy()
    lse, loss, dH, dW, _ = oracle.forward_backward(H, W, y)
    assert abs(loss - ref.item()) <= 1e-12 * max(1.0, abs(ref.item()))
    assert np.max(np.abs(lse - lse_ref)) <= 1e-12 * max(1.0, np.max(np.abs(lse_ref)))
    assert np.max(np.abs(dH - Ht.grad.numpy())) <= 1e-13
    assert np.max(np.abs(dW - Wt.grad.numpy())) <= 1e-13


def test_large_logits_are_stable():
    H, W, y = _rand(8, 5, 4, 9, w_scale=300.0)
    z = torch.tensor(H) @ torch.tensor(W).T
    lse, loss, _ = oracle.forward(H, W, y)
    assert np.all(np.isfinite(lse))
    assert np.max(np.abs(lse - torch.logsumexp(z, 1).numpy())) < 1e-9


def test_single_class_vocab_gives_zero_loss_and_gradients():
    H, W, _ = _rand(9, 6, 4, 1)
    y = np.zeros(6, dtype=np.int64)
    lse, loss, dH, dW, _ = oracle.forward_backward(H, W, y)
    assert np.max(np.abs(lse - (H @ W.T)[:, 0])) < 1e-14
    assert abs(loss) < 1e-14
    assert np.max(np.abs(dH)) < 1e-14 and np.max(np.abs(dW)) < 1e-14


def test_all_rows_ignored_gives_zero_loss_and_gradients():
    H, W, _ = _rand(10, 5, 4, 7)
    y = np.full(5, IGN, dtype=np.int64)
    lse, loss, dH, dW, count = oracle.forward_backward(H, W, y)
    assert count == 0 and loss == 0.0
    assert np.all(dH == 0.0) and np.all(dW == 0.0)
    assert np.max(np.abs(lse - torch.logsumexp(torch.tensor(H @ W.T), 1).numpy())) < 1e-13


def test_vocab_permutation_equivariance():
    H, W, y = _rand(11, 10, 6, 23, ignore=(2,))
    perm = np.random.default_rng(0).permutation(23)          # new row j holds old row perm[j]
    inv = np.argsort(perm)
    y2 = np.where(y == IGN, IGN, inv[np.where(y == IGN, 0, y)])
    lse, loss, dH, dW, _ = oracle.forward_backward(H, W, y)
    lse2, loss2, dH2, dW2, _ = oracle.forward_backward(H, W[perm], y2)
    assert abs(loss - loss2) < 1e-13
    assert np.max(np.abs(lse - lse2)) < 1e-13
    assert np.max(np.abs(dH - dH2)) < 1e-13
    assert np.max(np.abs(dW[perm] - dW2)) < 1e-13


def test_row_permutation_equivariance():
    H, W, y = _rand(12, 10, 6, 23, ignore=(2, 9))
    perm = np.random.default_rng(1).permutation(10)
    lse, loss, dH, dW, _ = oracle.forward_backward(H, W, y)
    lse2, loss2, dH2, dW2, _ = oracle.forward_backward(H[perm], W, y[perm])
    assert abs(loss - loss2) < 1e-13
    assert np.max(np.abs(lse[perm] - lse2)) < 1e-13
    assert np.max(np.abs(dH[perm] - dH2)) < 1e-13
    assert np.max(np.abs(dW - dW2)) < 1e-13


def test_grad_loss_scales_gradients_only():
    H, W, y = _rand(13, 8, 5, 19)
    _, l1, dH1, dW1, _ = oracle.forward_backward(H, W, y, grad_loss=1.0)
    _, l2, dH2, dW2, _ = oracle.forward_backward(H, W, y, grad_loss=-2.5)
    assert l1 == l2
    assert np.max(np.abs(dH2 + 2.5 * dH1)) < 1e-14
    assert np.max(np.abs(dW2 + 2.5 * dW1)) < 1e-14


def test_inner_product_identity():
    # <W, dW> = <H, dH> = sum_{n,v} dZ_nv z_nv: holds at any size, used for the
    # long-context parity check where dW cannot be sampled.
    H, W, y = _rand(14, 12, 7, 29, ignore=(3,))
    _, _, dH, dW, _ = oracle.forward_backward(H, W, y)
    assert abs(np.sum(W * dW) - np.sum(H * dH)) < 1e-13
    # Column sums of dW vanish: softmax and onehot both sum to one per row.
    assert np.max(np.abs(dW.sum(axis=0))) < 1e-13


def test_out_of_range_target_rejected():
    H, W, y = _rand(15, 3, 2, 5)
    y[1] = 5
    with pytest.raises(ValueError):
        oracle.forward(H, W, y)


def test_sampled_helpers_match_full_run():
    H, W, y = _rand(16, 40, 9, 70, ignore=(1, 2, 30))
    lse, _, dH, dW, _ = oracle.forward_backward(H, W, y, grad_loss=0.5)
    rows = np.array([0, 2, 17, 39])
    vocab_ids = np.array([0, 5, 69, int(y[0])])
    assert np.max(np.abs(oracle.lse_rows(H, W, rows) - lse[rows])) < 1e-13
    assert np.max(np.abs(oracle.dH_rows(H, W, y, rows, grad_loss=0.5) - dH[rows])) < 1e-14
    assert np.max(np.abs(oracle.dW_rows(H, W, y, lse, vocab_ids, grad_loss=0.5) - dW[vocab_ids])) < 1e-14


def test_filter_special_cases():
    H, W, y = _rand(17, 20, 6, 64, w_scale=2.0, ignore=(4,))
    full = oracle.forward_backward(H, W, y)
    f0 = oracle.forward_backward_filtered(H, W, y, 0.0, 8, 16)
    assert f0[5] == 0.0
    assert np.array_equal(f0[2], full[2]) or np.max(np.abs(f0[2] - full[2])) < 1e-15
    f_all = oracle.forward_backward_filtered(H, W, y, 2.0, 8, 16)
    assert f_all[5] == 1.0
    assert np.all(f_all[2] == 0.0) and np.all(f_all[3] == 0.0)
    fracs = [oracle.forward_backward_filtered(H, W, y, e, 8, 16)[5] for e in (1e-6, 1e-3, 1e-1)]
    assert fracs[0] <= fracs[1] <= fracs[2]
    # A skipped tile drops exactly its own terms: rows outside skipped tiles of
    # a one-row-tile filtering keep their exact dH.
    f1 = oracle.forward_backward_filtered(H, W, y, 1e-3, 1, 64)
    assert np.max(np.abs(f1[2] - full[2])) <= 1e-3 * np.max(np.abs(W)) * 64 / 19


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("with_bias", [False, True])
def test_general_form_matches_library_cross_entropy(reduction, with_bias):
    # Library cross-check of bias and reductions: F.linear + F.cross_entropy
    # on explicit fp64 logits, gradients by autograd.
    H, W, y = _rand(31, 13, 7, 29, w_scale=1.5, ignore=(2, 9))
    b = np.random.default_rng(5).standard_normal(29) if with_bias else None
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True) if with_bias else None
    z = torch.nn.functional.linear(Ht, Wt, bt)
    ref = torch.nn.functional.cross_entropy(z, torch.tensor(y), ignore_index=IGN, reduction=reduction)
    if reduction == "none":
        g = np.random.default_rng(6).standard_normal(13)
        ref.backward(torch.tensor(g))
    else:
        g = -0.75
        (ref * g).backward()
    out = oracle.forward_backward_ex(H, W, y, bias=b, reduction=reduction, grad=g)
    if reduction == "none":
        assert np.max(np.abs(out["loss"] - ref.detach().numpy())) < 1e-12
    else:
        assert abs(out["loss"] - ref.item()) < 1e-12
    assert np.max(np.abs(out["lse"] - torch.logsumexp(z.detach(), 1).numpy())) < 1e-12
    assert np.max(np.abs(out["dH"] - Ht.grad.numpy())) < 1e-13
    assert np.max(np.abs(out["dW"] - Wt.grad.numpy())) < 1e-13
    if with_bias:
        assert np.max(np.abs(out["db"] - bt.grad.numpy())) < 1e-13
    else:
        assert out["db"] is None


def test_general_form_bias_finite_differences():
    H, W, y = _rand(32, 5, 4, 9, w_scale=1.0, ignore=(1,))
    b = np.random.default_rng(7).standard_normal(9)
    out = oracle.forward_backward_ex(H, W, y, bias=b, reduction="sum", grad=1.0)
    h = 1e-6
    for v in range(9):
        bp, bm = b.copy(), b.copy()
        bp[v] += h
        bm[v] -= h
        fd = (oracle.forward_backward_ex(H, W, y, bias=bp, reduction="sum", need_grad=False)["loss"]
              - oracle.forward_backward_ex(H, W, y, bias=bm, reduction="sum", need_grad=False)["loss"]) / (2 * h)
        assert abs(fd - out["db"][v]) < 1e-6
    # db sums dZ over rows: the columns of dZ, not its rows, so sum_v db_v = 0.
    assert abs(out["db"].sum()) < 1e-13


def test_general_form_reduces_to_the_plain_mean():
    H, W, y = _rand(33, 11, 6, 17, ignore=(4,))
    a = oracle.forward_backward_ex(H, W, y, grad=2.0)
    lse, loss, dH, dW, _ = oracle.forward_backward(H, W, y, grad_loss=2.0)
    assert abs(a["loss"] - loss) < 1e-14
    assert np.max(np.abs(a["dH"] - dH)) < 1e-15 and np.max(np.abs(a["dW"] - dW)) < 1e-15


def test_filter_full_variants():
    H, W, y = _rand(34, 24, 6, 64, w_scale=2.0, ignore=(3,))
    full = oracle.forward_backward(H, W, y)
    f = oracle.forward_backward_filtered(H, W, y, 1e-3, 8, 16)
    fc = oracle.forward_backward_filtered(H, W, y, 1e-3, 8, 16, filter_dW=False)
    fe = oracle.forward_backward_filtered(H, W, y, 1e-3, 8, 16, filter_dH=False)
    assert np.array_equal(fc[2], f[2]) and np.max(np.abs(fc[3] - full[3])) < 1e-15
    assert np.array_equal(fe[3], f[3]) and np.max(np.abs(fe[2] - full[2])) < 1e-15


def test_filter_taller_dH_mask():
    H, W, y = _rand(35, 32, 6, 64, w_scale=2.0, ignore=(3,))
    a = oracle.forward_backward_filtered(H, W, y, 1e-3, 8, 16)
    b = oracle.forward_backward_filtered(H, W, y, 1e-3, 8, 16, dH_tile_rows=16)
    full = oracle.forward_backward(H, W, y)
    # dW and the skip statistic do not depend on the dH mask (dW up to the
    # fp64 summation order of the row blocks).
    assert np.max(np.abs(a[3] - b[3])) < 1e-15 and a[5] == b[5]
    # A taller dH mask drops a subset of what the 8-row mask drops, so its dH
    # is at least as close to the unfiltered one.
    assert np.max(np.abs(b[2] - full[2])) <= np.max(np.abs(a[2] - full[2])) + 1e-15
    c = oracle.forward_backward_filtered(H, W, y, 1e-3, 8, 16, dH_tile_rows=8)
    assert np.array_equal(a[2], c[2])
    with pytest.raises(ValueError):
        oracle.forward_backward_filtered(H, W, y, 1e-3, 8, 16, dH_tile_rows=12)


# ---- vocabulary sorting (Cut Cross-Entropy, Sec. 4.3 "Vocabulary sorting")

def test_average_logits_closed_forms():
    n, d, v = 9, 6, 17
    H, W, y = _rand(21, n, d, v, ignore=(0, 4, 7))
    valid = y != IGN
    # Linearity: the mean of z_nv over valid rows is W_v . mean(H_valid).
    a = oracle.average_logits(H, W, y)
    assert np.max(np.abs(a - W @ H[valid].mean(axis=0))) < 1e-13
    # A bias adds b_v to every logit, hence to the average.
    b = np.linspace(-2.0, 3.0, v)
    assert np.max(np.abs(oracle.average_logits(H, W, y, bias=b) - (a + b))) < 1e-13
    # W = 0: every logit is zero.
    assert np.all(oracle.average_logits(H, np.zeros_like(W), y) == 0.0)
    # No valid row: all zero.
    assert np.all(oracle.average_logits(H, W, np.full(n, IGN)) == 0.0)


def test_average_logits_ignore_ignored_rows():
    n, d, v = 8, 5, 11
    H, W, y = _rand(22, n, d, v, ignore=(1, 6))
    a = oracle.average_logits(H, W, y)
    H2 = H.copy()
    H2[[1, 6]] = 1e3 * np.arange(1, d + 1)
    assert np.array_equal(oracle.average_logits(H2, W, y), a)
    # Changing a valid row does move the average of every non-zero W row.
    H3 = H.copy()
    H3[2] += 1.0
    assert np.all(np.abs(oracle.average_logits(H3, W, y) - a) > 1e-6)


def test_average_logits_permute_with_the_vocabulary():
    n, d, v = 6, 4, 10
    H, W, y = _rand(23, n, d, v, ignore=(3,))
    perm = np.random.default_rng(5).permutation(v)
    inv = np.argsort(perm)
    y2 = np.where(y == IGN, IGN, inv[np.where(y == IGN, 0, y)])
    assert np.max(np.abs(oracle.average_logits(H, W[perm], y2) - oracle.average_logits(H, W, y)[perm])) < 1e-13


def test_vocabulary_order_is_descending_and_stable():
    a = np.array([0.5, 2.0, -1.0, 2.0, 0.5, 7.0, -0.0, 0.0, -1.0])
    order = oracle.vocabulary_order(a)
    brute = sorted(range(len(a)), key=lambda i: (-a[i], i))
    assert list(order) == brute
    assert list(order) == [5, 1, 3, 0, 4, 6, 7, 2, 8]


def _interleaved_case():
    # Even ids get a logit far below the rest for every row, odd ids sit
    # near zero: in id order every 2-wide column block mixes one of each.
    n, d, v = 6, 3, 8
    H = np.ones((n, d))
    H[:, 1] = np.linspace(-0.2, 0.2, n)
    W = np.zeros((v, d))
    W[0::2, 0] = -15.0
    W[1::2, 2] = np.linspace(0.1, 0.4, v // 2)
    y = np.array([1, 3, 5, 7, 1, IGN], dtype=np.int64)
    return H, W, y


def test_sorting_groups_negligible_columns_into_skippable_tiles():
    H, W, y = _interleaved_case()
    eps = 2.0 ** -12
    *_, frac_id = oracle.forward_backward_filtered(H, W, y, eps, 3, 2)
    order = oracle.vocabulary_order(oracle.average_logits(H, W, y))
    assert sorted(order[:4]) == [1, 3, 5, 7]
    lse, loss, dH, dW, count, frac_sorted = oracle.forward_backward_filtered(H, W, y, eps, 3, 2, vocab_order=order)
    assert frac_id == 0.0
    assert frac_sorted == 0.5          # the two all-even column blocks, both row blocks
    # The skipped G are all below eps, so the result stays within the filter's error bound.
    ref = oracle.forward_backward(H, W, y)
    assert abs(loss - ref[1]) < 1e-15 and np.max(np.abs(lse - ref[0])) < 1e-15
    assert np.max(np.abs(dH - ref[2])) < 2 * eps * 15 and np.max(np.abs(dW - ref[3])) < 2 * eps
    assert not np.array_equal(dW, ref[3])


def test_vocab_order_equivariance_and_degenerate_cases():
    n, d, v = 10, 4, 12
    H, W, y = _rand(24, n, d, v, w_scale=2.0, ignore=(2, 9))
    eps = 0.01
    perm = np.random.default_rng(6).permutation(v)
    # Identity order is the plain tile mask.
    a = oracle.forward_backward_filtered(H, W, y, eps, 4, 3)
    b = oracle.forward_backward_filtered(H, W, y, eps, 4, 3, vocab_order=np.arange(v))
    for x, z in zip(a, b):
        assert np.array_equal(np.asarray(x), np.asarray(z))
    # Sorting by `perm` equals relabelling the vocabulary by hand.
    inv = np.argsort(perm)
    y2 = np.where(y == IGN, IGN, inv[np.where(y == IGN, 0, y)])
    hand = oracle.forward_backward_filtered(H, W[perm], y2, eps, 4, 3)
    got = oracle.forward_backward_filtered(H, W, y, eps, 4, 3, vocab_order=perm)
    assert got[5] == hand[5]
    assert np.max(np.abs(got[2] - hand[2])) < 1e-13
    assert np.max(np.abs(got[3][perm] - hand[3])) < 1e-13
    # eps = 0 filters nothing: any order gives the unfiltered result.
    ref = oracle.forward_backward(H, W, y)
    got0 = oracle.forward_backward_filtered(H, W, y, 0.0, 4, 3, vocab_order=perm)
    assert got0[5] == 0.0
    assert np.max(np.abs(got0[2] - ref[2])) < 1e-13 and np.max(np.abs(got0[3] - ref[3])) < 1e-13
    with pytest.raises(ValueError):
        oracle.forward_backward_filtered(H, W, y, eps, 4, 3, vocab_order=np.zeros(v, dtype=np.int64))


def test_vocab_order_with_ignore_index_inside_the_vocabulary():
    n, d, v = 8, 4, 9
    H, W, _ = _rand(25, n, d, v)
    y = np.array([0, 4, 4, 8, 2, 4, 1, 7], dtype=np.int64)      # 4 is the ignore index
    perm = np.random.default_rng(7).permutation(v)
    ref = oracle.forward_backward(H, W, y, ignore_index=4)
    got = oracle.forward_backward_filtered(H, W, y, 0.0, 4, 3, ignore_index=4, vocab_order=perm)
    assert got[4] == ref[4] == 5
    assert abs(got[1] - ref[1]) < 1e-14
    assert np.max(np.abs(got[2] - ref[2])) < 1e-13 and np.max(np.abs(got[3] - ref[3])) < 1e-13


# ---- AdamW fused into the weight gradient (FORGE explainer, Sec. 2)

_HP = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1}


def test_adamw_matches_torch_optim_over_several_steps():
    rng = np.random.default_rng(31)
    p0 = rng.standard_normal((7, 5))
    grads = [rng.standard_normal((7, 5)) for _ in range(4)]
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=_HP["lr"], betas=(_HP["beta1"], _HP["beta2"]), eps=_HP["eps"],
                            weight_decay=_HP["weight_decay"])
    p, m, v = p0, np.zeros_like(p0), np.zeros_like(p0)
    for t, g in enumerate(grads, start=1):
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = oracle.adamw_step(p, g, m, v, t, **_HP)
        assert np.max(np.abs(p - tp.detach().numpy())) < 1e-15
    st = opt.state[tp]
    assert np.max(np.abs(m - st["exp_avg"].numpy())) < 1e-15
    assert np.max(np.abs(v - st["exp_avg_sq"].numpy())) < 1e-15


def test_adamw_first_step_closed_form():
    # From zero moments the bias-corrected ratio is g / (|g| + eps).
    rng = np.random.default_rng(32)
    p0, g = rng.standard_normal(20), rng.standard_normal(20)
    p, m, v = oracle.adamw_step(p0, g, np.zeros(20), np.zeros(20), 1, **_HP)
    lr, wd, eps = _HP["lr"], _HP["weight_decay"], _HP["eps"]
    assert np.max(np.abs(p - (p0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps)))) < 1e-15
    assert np.max(np.abs(m - (1 - _HP["beta1"]) * g)) < 1e-15
    assert np.max(np.abs(v - (1 - _HP["beta2"]) * g * g)) < 1e-15
    # No learning rate: the parameters stay; the moments still move.
    p2, m2, _ = oracle.adamw_step(p0, g, np.zeros(20), np.zeros(20), 1, **{**_HP, "lr": 0.0})
    assert np.array_equal(p2, p0) and np.any(m2 != 0)
    with pytest.raises(ValueError):
        oracle.adamw_step(p0, g, m, v, 0, **_HP)


def test_fused_step_equals_gradient_then_optimizer():
    n, d, v = 9, 6, 13
    H, W, y = _rand(33, n, d, v, ignore=(4,))
    rng = np.random.default_rng(34)
    master, m0, v0 = W + 1e-3 * rng.standard_normal(W.shape), rng.standard_normal(W.shape), rng.random(W.shape)
    hp = {**_HP, "step": 3}
    r = oracle.forward_backward_adamw(H, W, y, master, m0, v0, hp, grad_loss=0.5)
    lse, loss, dH, dW, count = oracle.forward_backward(H, W, y, grad_loss=0.5)
    # dW of a library autograd pass, then the library optimizer.
    Wt = torch.tensor(W, requires_grad=True)
    ce = torch.nn.functional.cross_entropy(torch.tensor(H) @ Wt.T, torch.tensor(y), ignore_index=IGN) * 0.5
    ce.backward()
    assert np.max(np.abs(Wt.grad.numpy() - dW)) < 1e-14
    tp = torch.tensor(master, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                            weight_decay=hp["weight_decay"])
    opt.state[tp] = {"step": torch.tensor(2.0, dtype=torch.float64), "exp_avg": torch.tensor(m0),
                     "exp_avg_sq": torch.tensor(v0)}
    tp.grad = Wt.grad
    opt.step()
    assert np.max(np.abs(r["master"] - tp.detach().numpy())) < 1e-14
    assert r["count"] == count and abs(r["loss"] - loss) < 1e-15


# ---------------------------------------------------------------- input widening
# Every parity test feeds both sides the same bf16 inputs and the oracle widens
# them to fp64 (inputs_f64). These pins check that widening against two
# decoders that share nothing with it: torch's own bfloat16 -> float64
# conversion, and the bf16 format written out with integers (1 sign bit,
# 8 exponent bits with bias 127, 7 fraction bits; subnormals at exponent 0).

def _decode_bf16_by_fields(bits: int) -> float:
    sign = -1.0 if bits & 0x8000 else 1.0
    exp = (bits >> 7) & 0xFF
    frac = bits & 0x7F
    if exp == 0xFF:
        assert frac == 0, "NaN patterns are not decoded here"
        return sign * math.inf
    if exp == 0:
        return sign * math.ldexp(frac / 128.0, -126)
    return sign * math.ldexp(1.0 + frac / 128.0, exp - 127)


def _all_non_nan_bf16_patterns() -> np.ndarray:
    bits = np.arange(1 << 16, dtype=np.uint32)
    exp = (bits >> 7) & 0xFF
    frac = bits & 0x7F
    return bits[~((exp == 0xFF) & (frac != 0))].astype(np.uint16)


def test_inputs_f64_matches_torch_on_every_bf16_pattern():
    bits = _all_non_nan_bf16_patterns()
    assert bits.size == (1 << 16) - 2 * 127     # NaNs excluded, both infinities kept
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    h64, w64 = oracle.inputs_f64(bits.reshape(2, -1), bits[::-1].reshape(-1, 2))
    assert h64.dtype == np.float64 and w64.dtype == np.float64
    assert h64.shape == (2, bits.size // 2) and w64.shape == (bits.size // 2, 2)
    np.testing.assert_array_equal(h64.ravel(), ref)
    np.testing.assert_array_equal(w64.ravel(), ref[::-1])     # the second array is W's, not H's again
    assert np.array_equal(np.signbit(h64.ravel()), np.signbit(ref))   # -0 stays -0


def test_inputs_f64_matches_the_bit_fields_on_every_bf16_pattern():
    bits = _all_non_nan_bf16_patterns()
    ref = np.array([_decode_bf16_by_fields(int(b)) for b in bits], dtype=np.float64)
    got, _ = oracle.inputs_f64(bits, bits[:1])
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xBF80, -1.0), (0x4000, 2.0), (0x3F00, 0.5), (0x3FC0, 1.5),
    (0x0001, 2.0 ** -133),                     # smallest subnormal
    (0x0080, 2.0 ** -126),                     # smallest normal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),  # largest finite
    (0x7F80, math.inf), (0xFF80, -math.inf), (0x8000, -0.0), (0x0000, 0.0),
])
def test_inputs_f64_known_values(bits, value):
    got, _ = oracle.inputs_f64(np.array([bits], dtype=np.uint16), np.zeros(1, dtype=np.uint16))
    assert got[0] == value and math.copysign(1.0, got[0]) == math.copysign(1.0, value)
