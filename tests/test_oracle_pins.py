"""Pins for the fp64 oracle, each against something other than the oracle itself.

* brute force written with modular arithmetic per token (no roll or partition tensors);
* library special cases: ``numpy.roll``, reshape-based partition, ``torch`` SDPA in fp64
  on the CPU (forward) and ``torch.autograd`` through it (backward);
* invariants (identities, row sums, index-map counts and symmetry, constant V,
  permutation equivariance, the shift mask as a "which tokens wrapped" test);
* closed forms (a 1x1 window returns V; a fully masked 2x2 window returns each V up to
  an e^-100 leak) and central finite differences of the backward.

The method follows the NVIDIA Swin talk transcript (uticex.com, article 1598): section 1
(window attention, window shift, relative position bias), section 2 (shift, partition
and reverse as index mappings; mask and bias as tensors) and section 3 (bias lookup done
once ahead of the attention).
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _table(M, nH, seed):
    return _rand(((2 * M - 1) ** 2, nH), seed, 0.5)


# ---------------------------------------------------------------------------------
# brute force: every original token, its rolled position, its window, its keys
# ---------------------------------------------------------------------------------

def _region(c, L, M, s):
    if c < L - M:
        return 0
    if c < L - s:
        return 1
    return 2


def brute_force_fwd(qkv, table, nH, M, s):
    B, H, W, C3 = qkv.shape
    C = C3 // 3
    hd = C // nH
    Y = np.zeros((B, H, W, C))
    for b, y, x in itertools.product(range(B), range(H), range(W)):
        ry, rx = (y - s) % H, (x - s) % W          # where token (y, x) sits after the shift
        wy, wx = ry // M, rx // M
        liy, lix = ry % M, rx % M
        lab = 3 * _region(ry, H, M, s) + _region(rx, W, M, s)
        keys = []
        for ly, lx in itertools.product(range(M), range(M)):
            kry, krx = wy * M + ly, wx * M + lx
            klab = 3 * _region(kry, H, M, s) + _region(krx, W, M, s)
            keys.append(((kry + s) % H, (krx + s) % W, ly, lx, klab))
        for h in range(nH):
            q = qkv[b, y, x, h * hd:(h + 1) * hd]
            logits, vals = [], []
            for (ky, kx, ly, lx, klab) in keys:
                k = qkv[b, ky, kx, C + h * hd:C + (h + 1) * hd]
                r = (liy - ly + M - 1) * (2 * M - 1) + (lix - lx + M - 1)
                z = float(q @ k) / math.sqrt(hd) + table[r, h] + (0.0 if klab == lab else -100.0)
                logits.append(z)
                vals.append(qkv[b, ky, kx, 2 * C + h * hd:2 * C + (h + 1) * hd])
            logits = np.array(logits)
            p = np.exp(logits - logits.max())
            p /= p.sum()
            Y[b, y, x, h * hd:(h + 1) * hd] = p @ np.array(vals)
    return Y


BRUTE_CASES = [
    # (B, H, W, C, nH, M, s)
    (1, 8, 8, 8, 2, 4, 2),    # the tiny workload's geometry with a narrow head
    (1, 4, 4, 6, 2, 2, 1),
    (2, 8, 8, 4, 1, 2, 0),
    (1, 8, 8, 4, 1, 2, 1),
    (1, 12, 12, 4, 2, 4, 0),
    (1, 12, 12, 4, 2, 4, 1),
    (1, 12, 12, 4, 2, 4, 3),
    (1, 4, 4, 4, 1, 4, 3),    # one window, shift inside it
    (1, 8, 12, 6, 3, 4, 2),   # non-square grid
]


@pytest.mark.parametrize("B,H,W,C,nH,M,s", BRUTE_CASES)
def test_fwd_matches_brute_force(oracle_mod, B, H, W, C, nH, M, s):
    qkv = _rand((B, H, W, 3 * C), 1 + H + M + s)
    table = _table(M, nH, 7 + s)
    Y = oracle_mod.fwd(qkv, table, nH, M, s)
    Yb = brute_force_fwd(qkv, table, nH, M, s)
    assert np.abs(Y - Yb).max() < 1e-12


def test_tiny_workload_full_head_width_matches_brute_force(oracle_mod):
    from swin_window_attention_gb300 import inputs
    wl = inputs.BY_NAME["tiny"]
    qkv = inputs.act_f64(inputs.make_qkv(wl))
    table = inputs.make_table(wl).double().numpy()
    Y = oracle_mod.fwd(qkv, table, wl.nH, wl.M, wl.s)
    assert np.abs(Y - brute_force_fwd(qkv, table, wl.nH, wl.M, wl.s)).max() < 1e-12


# ---------------------------------------------------------------------------------
# index mappings against library routines and as identities
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("s", [0, 1, 3, 5])
def test_roll_is_numpy_roll_and_unroll_inverts(oracle_mod, s):
    x = _rand((2, 10, 15, 3), s)
    r = oracle_mod.roll(x, s)
    assert np.array_equal(r, np.roll(x, shift=(-s, -s), axis=(1, 2)))
    assert np.array_equal(oracle_mod.unroll(r, s), x)
    assert np.array_equal(oracle_mod.roll(oracle_mod.unroll(x, s), s), x)


@pytest.mark.parametrize("H,W,M", [(8, 8, 4), (14, 21, 7), (12, 24, 12), (6, 6, 1)])
def test_partition_is_reshape_and_reverse_inverts(oracle_mod, H, W, M):
    x = _rand((2, H, W, 5), H * W)
    p = oracle_mod.partition(x, M)
    ref = x.reshape(2, H // M, M, W // M, M, 5).transpose(0, 1, 3, 2, 4, 5).reshape(
        2, (H // M) * (W // M), M * M, 5)
    assert np.array_equal(p, ref)
    assert np.array_equal(oracle_mod.reverse(p, H, W, M), x)


@pytest.mark.parametrize("H,W,M,s", [(8, 8, 4, 2), (56, 56, 7, 3), (12, 12, 12, 6), (14, 28, 7, 0)])
def test_gather_map_is_a_permutation_read_once(oracle_mod, H, W, M, s):
    g = oracle_mod.gather(H, W, M, s)
    assert sorted(g.ravel().tolist()) == list(range(H * W))
    # token read by window w slot i: rolled position (wy*M+ly, wx*M+lx) + s
    nWx = W // M
    w, i = 1 % g.shape[0], M * M - 1
    wy, wx = w // nWx, w % nWx
    y, x = (wy * M + M - 1 + s) % H, (wx * M + M - 1 + s) % W
    assert g[w, i] == y * W + x


@pytest.mark.parametrize("M", [1, 2, 4, 7, 12])
def test_relidx_counts_centre_symmetry(oracle_mod, M):
    idx = oracle_mod.relidx(M)
    N, R = M * M, (2 * M - 1) ** 2
    assert idx.min() == 0 and idx.max() == R - 1
    assert np.all(np.diag(idx) == (R - 1) // 2)
    assert np.all(idx + idx.T == R - 1)
    counts = np.bincount(idx.ravel(), minlength=R).reshape(2 * M - 1, 2 * M - 1)
    for a, b in itertools.product(range(2 * M - 1), repeat=2):
        assert counts[a, b] == (M - abs(a - (M - 1))) * (M - abs(b - (M - 1)))
    # along a row of the window (same y), the index moves by one per step in x
    if M > 1:
        assert idx[0, 1] == idx[0, 0] - 1 and idx[0, M] == idx[0, 0] - (2 * M - 1)


def test_dense_bias_is_a_table_lookup(oracle_mod):
    M, nH = 4, 3
    table = _table(M, nH, 3)
    db = oracle_mod.dense_bias(table, nH, M)
    idx = oracle_mod.relidx(M)
    assert np.array_equal(db, np.transpose(table[idx], (2, 0, 1)))


@pytest.mark.parametrize("H,W,M,s", [(8, 8, 4, 2), (56, 56, 7, 3), (28, 14, 7, 3),
                                     (12, 12, 12, 6), (96, 96, 12, 6), (8, 8, 4, 0), (7, 7, 7, 0)])
def test_mask_is_the_wrapped_token_test(oracle_mod, H, W, M, s):
    """Two tokens of one window are masked iff, along some axis, exactly one of them came
    from the far side of the image through the cyclic shift."""
    mk = oracle_mod.mask(H, W, M, s)
    assert set(np.unique(mk).tolist()) <= {0.0, -100.0}
    if s == 0:
        assert not mk.any()
    nWx, N = W // M, M * M
    for w in range(mk.shape[0]):
        wy, wx = w // nWx, w % nWx
        ry = wy * M + np.arange(N) // M
        rx = wx * M + np.arange(N) % M
        wrap_y, wrap_x = ry >= H - s, rx >= W - s
        diff = (wrap_y[:, None] != wrap_y[None, :]) | (wrap_x[:, None] != wrap_x[None, :])
        assert np.array_equal(mk[w], np.where(diff, -100.0, 0.0))
        assert np.all(np.diag(mk[w]) == 0)


# ---------------------------------------------------------------------------------
# attention invariants
# ---------------------------------------------------------------------------------

def test_probability_rows_sum_to_one(oracle_mod):
    H = W = 8
    M, s, nH, C = 4, 2, 2, 16
    qkv = _rand((1, H, W, 3 * C), 5, 2.0)
    table = _table(M, nH, 5)
    for w in range(4):
        for h in range(nH):
            P = oracle_mod.probs(qkv, table, nH, M, s, 0, w, h)
            assert np.all(P >= 0)
            assert np.abs(P.sum(1) - 1).max() < 1e-14


def test_constant_v_gives_that_constant(oracle_mod):
    B, H, W, C, nH, M, s = 2, 8, 8, 8, 2, 4, 2
    qkv = _rand((B, H, W, 3 * C), 9)
    const = _rand((C,), 10)
    qkv[..., 2 * C:] = const
    Y = oracle_mod.fwd(qkv, _table(M, nH, 1), nH, M, s)
    assert np.abs(Y - const).max() < 1e-13


def test_window_size_one_returns_v(oracle_mod):
    """M = 1: each window holds one token, so the softmax is exactly 1 and Y is V with
    heads concatenated in channel order (checks the q/k/v channel split)."""
    qkv = _rand((2, 3, 5, 12), 11)
    Y = oracle_mod.fwd(qkv, _table(1, 2, 2), 2, 1, 0)
    assert np.array_equal(Y, qkv[..., 8:])


def test_fully_masked_two_by_two_window_closed_form(oracle_mod):
    """H = W = M = 2, s = 1: all four tokens wrap differently, so every off-diagonal
    pair is masked. With q = k = 0 and a zero table the logits are 0 on the diagonal and
    -100 elsewhere: Y_i = (v_i + e^-100 * sum_{j != i} v_j) / (1 + 3 e^-100)."""
    C = 4
    qkv = np.zeros((1, 2, 2, 3 * C))
    v = _rand((1, 2, 2, C), 12)
    qkv[..., 2 * C:] = v
    Y = oracle_mod.fwd(qkv, np.zeros((9, 1)), 1, 2, 1)
    e = math.exp(-100.0)
    tot = v.sum(axis=(1, 2), keepdims=True)
    expect = (v + e * (tot - v)) / (1 + 3 * e)
    assert np.abs(Y - expect).max() < 1e-15


def test_permuting_tokens_inside_an_unshifted_window_permutes_outputs(oracle_mod):
    H = W = M = 4
    C, nH = 8, 2
    qkv = _rand((1, H, W, 3 * C), 13)
    Y = oracle_mod.fwd(qkv, np.zeros(((2 * M - 1) ** 2, nH)), nH, M, 0)
    perm = np.random.default_rng(1).permutation(H * W)
    qp = qkv.reshape(1, H * W, 3 * C)[:, perm].reshape(1, H, W, 3 * C)
    Yp = oracle_mod.fwd(qp, np.zeros(((2 * M - 1) ** 2, nH)), nH, M, 0)
    assert np.abs(Yp.reshape(1, H * W, C) - Y.reshape(1, H * W, C)[:, perm]).max() < 1e-13


def test_shift_zero_equals_plain_window_attention(oracle_mod):
    B, H, W, C, nH, M = 2, 14, 21, 12, 3, 7
    hd = C // nH
    qkv = _rand((B, H, W, 3 * C), 14)
    table = _table(M, nH, 14)
    Y = oracle_mod.fwd(qkv, table, nH, M, 0)
    t = torch.from_numpy(qkv).view(B, H // M, M, W // M, M, 3, nH, hd)
    t = t.permute(5, 0, 1, 3, 6, 2, 4, 7).reshape(3, B, -1, nH, M * M, hd)
    q, k, v = t[0], t[1], t[2]
    db = torch.from_numpy(oracle_mod.dense_bias(table, nH, M))
    a = torch.softmax(q @ k.transpose(-1, -2) / math.sqrt(hd) + db, dim=-1) @ v
    a = a.view(B, H // M, W // M, nH, M, M, hd).permute(0, 1, 4, 2, 5, 3, 6).reshape(B, H, W, C)
    assert np.abs(Y - a.numpy()).max() < 1e-12


def test_single_window_zero_bias_is_global_attention(oracle_mod):
    B, H, C, nH = 2, 7, 64, 2
    hd = C // nH
    qkv = _rand((B, H, H, 3 * C), 15)
    Y = oracle_mod.fwd(qkv, np.zeros(((2 * H - 1) ** 2, nH)), nH, H, 0)
    t = torch.from_numpy(qkv).view(B, H * H, 3, nH, hd).permute(2, 0, 3, 1, 4)
    o = F.scaled_dot_product_attention(t[0], t[1], t[2])
    o = o.permute(0, 2, 1, 3).reshape(B, H, H, C)
    assert np.abs(Y - o.numpy()).max() < 1e-12


# ---------------------------------------------------------------------------------
# the whole path against torch (fp64, CPU): roll + reshape + SDPA, autograd backward
# ---------------------------------------------------------------------------------

def torch_swin_attention(qkv, table, nH, M, s):
    B, H, W, C3 = qkv.shape
    C = C3 // 3
    hd, N, nWy, nWx = C // nH, M * M, H // M, W // M
    x = torch.roll(qkv, shifts=(-s, -s), dims=(1, 2))
    x = x.view(B, nWy, M, nWx, M, 3, nH, hd).permute(5, 0, 1, 3, 6, 2, 4, 7)
    x = x.reshape(3, B, nWy * nWx, nH, N, hd)
    ly, lx = torch.meshgrid(torch.arange(M), torch.arange(M), indexing="ij")
    ly, lx = ly.reshape(-1), lx.reshape(-1)
    rel = (ly[:, None] - ly[None, :] + M - 1) * (2 * M - 1) + (lx[:, None] - lx[None, :] + M - 1)
    bias = table[rel.reshape(-1)].view(N, N, nH).permute(2, 0, 1)
    wy = torch.arange(nWy).repeat_interleave(nWx)
    wx = torch.arange(nWx).repeat(nWy)
    ry = wy[:, None] * M + ly[None, :]
    rx = wx[:, None] * M + lx[None, :]
    wrap_y, wrap_x = ry >= H - s, rx >= W - s
    diff = (wrap_y[:, :, None] != wrap_y[:, None, :]) | (wrap_x[:, :, None] != wrap_x[:, None, :])
    maskt = torch.where(diff, -100.0, 0.0).to(qkv.dtype) if s > 0 else torch.zeros(
        nWy * nWx, N, N, dtype=qkv.dtype)
    attn_mask = bias[None, None] + maskt[None, :, None]
    o = F.scaled_dot_product_attention(x[0], x[1], x[2], attn_mask=attn_mask)
    o = o.view(B, nWy, nWx, nH, M, M, hd).permute(0, 1, 4, 2, 5, 3, 6).reshape(B, H, W, C)
    return torch.roll(o, shifts=(s, s), dims=(1, 2))


@pytest.mark.parametrize("B,H,W,C,nH,M,s", [
    (2, 8, 8, 64, 2, 4, 2),
    (1, 14, 14, 64, 2, 7, 3),
    (1, 24, 24, 32, 1, 12, 6),
    (1, 7, 7, 64, 2, 7, 0),
    (2, 14, 28, 32, 1, 7, 3),
])
def test_fwd_bwd_match_torch_sdpa_autograd(oracle_mod, B, H, W, C, nH, M, s):
    qkv = _rand((B, H, W, 3 * C), 20 + M)
    table = _table(M, nH, 21 + M) * 0.1
    G = _rand((B, H, W, C), 22 + M)
    tq = torch.from_numpy(qkv).requires_grad_(True)
    tt = torch.from_numpy(table).requires_grad_(True)
    Yt = torch_swin_attention(tq, tt, nH, M, s)
    (Yt * torch.from_numpy(G)).sum().backward()
    Y = oracle_mod.fwd(qkv, table, nH, M, s)
    dqkv, dtab = oracle_mod.bwd(qkv, G, table, nH, M, s)
    assert np.abs(Y - Yt.detach().numpy()).max() < 1e-11
    assert np.abs(dqkv - tq.grad.numpy()).max() < 1e-10
    assert np.abs(dtab - tt.grad.numpy()).max() < 1e-9


# ---------------------------------------------------------------------------------
# backward against central finite differences
# ---------------------------------------------------------------------------------

def test_bwd_matches_finite_differences(oracle_mod):
    B, H, W, C, nH, M, s = 1, 8, 8, 8, 2, 4, 2
    qkv = _rand((B, H, W, 3 * C), 30)
    table = _table(M, nH, 31)
    G = _rand((B, H, W, C), 32)
    dqkv, dtab = oracle_mod.bwd(qkv, G, table, nH, M, s)
    L = lambda q, t: float((oracle_mod.fwd(q, t, nH, M, s) * G).sum())  # noqa: E731
    eps = 1e-6
    rng = np.random.default_rng(33)
    for _ in range(24):
        e = tuple(int(rng.integers(0, n)) for n in qkv.shape)
        qp, qm = qkv.copy(), qkv.copy()
        qp[e] += eps
        qm[e] -= eps
        fd = (L(qp, table) - L(qm, table)) / (2 * eps)
        assert abs(fd - dqkv[e]) <= 1e-6 * max(1.0, abs(fd))
    for r in range(table.shape[0]):
        for h in range(nH):
            tp, tm = table.copy(), table.copy()
            tp[r, h] += eps
            tm[r, h] -= eps
            fd = (L(qkv, tp) - L(qkv, tm)) / (2 * eps)
            assert abs(fd - dtab[r, h]) <= 1e-6 * max(1.0, abs(fd))
