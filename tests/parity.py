"""Helpers shared by the GPU parity tests: uploads, state read-back and the
acceptance rules (bit-exact state and gather; logits within
1e-2 * max|oracle logit| per row; the top-k rule with that tolerance)."""

from __future__ import annotations

import numpy as np
import torch

import oracle

LOGIT_RTOL = 1e-2  # |gpu - oracle| <= LOGIT_RTOL * max_j |oracle[r, j]| per row


def dev_i32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def dev_f32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def dev_bf16(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(device)


def read_active(h, seq):
    act, cnt, bm, packed = h.get_active(seq)
    m = int(cnt.item())
    return m, act[:m].cpu().numpy(), bm.cpu().numpy().view(np.uint32)


def check_state(h, seq, ost: oracle.OracleStream, full: bool = True):
    """I_t, count, bitmap and |S| bit-exact; with full=True also ring and counts."""
    I = ost.active()
    m, act, bm = read_active(h, seq)
    assert m == len(I), f"|I_t| {m} != {len(I)}"
    assert np.array_equal(act, I), "I_t differs"
    assert np.array_equal(bm, oracle.bitmap_words(I, ost.V)), "bitmap differs"
    ring, length, counts = h.get_state(seq)
    S = ost.S
    assert int(length.item()) == len(S), "stream length differs"
    if full:
        W = ost.W_max
        ring = ring.cpu().numpy()
        start = max(0, len(S) - W)
        for p in range(start, len(S)):
            assert ring[p % W] == S[p], f"ring slot of position {p}"
        want = np.bincount(np.asarray(S[start:], dtype=np.int64), minlength=ost.V)
        assert np.array_equal(counts.cpu().numpy().astype(np.int64), want), "window counts differ"
    return I


def check_packed(h, seq, W_bits, I):
    _, _, _, packed = h.get_active(seq)
    got = packed[: len(I)].cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.gather_rows(W_bits, I)), "packed sub-head differs"


def check_logits(got, want):
    got = np.asarray(got, dtype=np.float32)
    tol = LOGIT_RTOL * np.abs(want).max(axis=1, keepdims=True)
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} logits out of tolerance (max err {err.max():.3g})"
    return tol[:, 0]


def check_topk(ids, vals, want, I, k, tol):
    """Top-k rule.  For each rank p the GPU id equals the oracle id, or the two
    ids' oracle logits are within tol of each other; every GPU id is in I_t,
    distinct, and has an oracle logit >= the oracle's k-th best - tol; GPU
    values match the oracle logits of the GPU ids within tol; rows with fewer
    than k active ids are padded with (-1, -inf)."""
    ids = np.asarray(ids)
    vals = np.asarray(vals)
    I = np.asarray(I)
    n, m = want.shape
    kk = min(k, m)
    o_ids, o_vals = oracle.topk_remap(want, I, k)
    pos = {int(g): j for j, g in enumerate(I.tolist())}
    for r in range(n):
        assert np.all(ids[r, kk:] == -1) and np.all(np.isneginf(vals[r, kk:])), "padding"
        got = [int(x) for x in ids[r, :kk]]
        assert len(set(got)) == kk, f"row {r}: repeated ids"
        assert all(g in pos for g in got), f"row {r}: id outside I_t"
        L = lambda g: float(want[r, pos[g]])  # noqa: E731
        for p in range(kk):
            if got[p] != int(o_ids[r, p]):
                assert abs(L(got[p]) - L(int(o_ids[r, p]))) <= tol[r], f"row {r} rank {p}: id mismatch"
        thr = float(o_vals[r, kk - 1]) - tol[r] if kk > 0 else -np.inf
        assert all(L(g) >= thr for g in got), f"row {r}: id below the k-th best"
        assert all(abs(float(vals[r, p]) - L(got[p])) <= tol[r] for p in range(kk)), f"row {r}: values"


def check_projection(logits_dev, ids_dev, vals_dev, hid_bits, W_bits, I, k):
    """Logits (first |I| columns) and top-k against the oracle."""
    I = np.asarray(I)
    want = oracle.project(hid_bits, oracle.gather_rows(W_bits, I))
    got = logits_dev[:, : len(I)].cpu().numpy()
    tol = check_logits(got, want)
    check_topk(ids_dev.cpu().numpy(), vals_dev.cpu().numpy(), want, I, k, tol)
    return want
