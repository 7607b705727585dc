"""Pins of the CPU oracle to things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong tie-break or window edge)
fails at least one test:

* hand-worked toy streams (tests/golden/toy_streams.json), derived by hand
  from the formal definitions of MicroSpec §3.2;
* brute force on tiny inputs (Top-K by a full Python sort; the window by an
  independent incremental occurrence-count implementation);
* exact-arithmetic projections (small integers times powers of two, summed
  with Python integers);
* invariants of I_t and special cases the definitions fix.
"""

import json
import os
import math
import random

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "toy_streams.json")


def _load():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Hand-worked toys
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("toy", _load()["toys"], ids=lambda t: t["name"])
def test_toy_streams(toy):
    V, W = toy["V"], toy["W_max"]
    Z = None if toy["prefill_logits"] is None else np.array(toy["prefill_logits"], np.float32)
    S = O.stream_init(toy["prompt"], Z, toy["K_pre"])
    assert S == toy["S_init"]
    assert O.active_vocab(S, W).tolist() == toy["I_init"]
    for st in toy["steps"]:
        assert O.draft_candidates(st["tree"]) == st["C_draft"]
        zv = None
        if toy["K_ver"] > 0:
            zv = np.array(st["verify"], np.float32)[st["verify_row"]]
            assert O.top_k(zv, toy["K_ver"]) == st["C_ver"]
        S = O.stream_append(S, st["tree"], zv, toy["K_ver"])
        assert S == st["S"]
        I = O.active_vocab(S, W)
        assert I.tolist() == st["I"]
        if "bitmap" in st:
            assert O.bitmap_words(I, V).tolist() == st["bitmap"]


def test_toy_through_state_holder():
    toy = _load()["toys"][0]
    st = O.OracleStream(toy["V"], toy["W_max"], toy["K_pre"], toy["K_ver"])
    st.init(toy["prompt"], np.array(toy["prefill_logits"], np.float32))
    for s in toy["steps"]:
        st.append(s["tree"], np.array(s["verify"], np.float32), s["verify_row"])
        assert st.active().tolist() == s["I"]
    assert st.bitmap().tolist() == toy["steps"][-1]["bitmap"]


@pytest.mark.parametrize("case", _load()["bitmaps"])
def test_bitmap_golden(case):
    assert O.bitmap_words(case["I"], case["V"]).tolist() == case["words"]


# ---------------------------------------------------------------------------
# Top-K against brute force
# ---------------------------------------------------------------------------
def _brute_topk(z, K):
    return sorted(range(len(z)), key=lambda i: (-float(z[i]), i))[:K]


def test_topk_brute_force_with_ties():
    rng = random.Random(1234)
    for _ in range(300):
        V = rng.randint(1, 40)
        K = rng.randint(0, V + 2)
        z = np.array([rng.choice([-1.5, 0.0, 0.25, 2.0, 3.0]) for _ in range(V)], np.float32)
        assert O.top_k(z, K) == _brute_topk(z, K)


def test_topk_rows_match_per_row():
    rng = np.random.default_rng(5)
    Z = rng.integers(-3, 4, size=(17, 23)).astype(np.float32)
    T = O.top_k_rows(Z, 5)
    for r in range(Z.shape[0]):
        assert T[r].tolist() == _brute_topk(Z[r], 5)


def test_topk_signed_zero_is_a_tie():
    z = np.array([-0.0, 0.0, -1.0], np.float32)
    assert O.top_k(z, 2) == [0, 1]


def _brute_topk_nan(z, K):
    """First K of a stable descending sort of the non-NaN entries."""
    return sorted((i for i in range(len(z)) if not math.isnan(float(z[i]))), key=lambda i: (-float(z[i]), i))[:K]


def test_topk_nan_never_ranks_and_infinities_order():
    rng = random.Random(99)
    for _ in range(300):
        V = rng.randint(1, 30)
        K = rng.randint(0, V + 2)
        z = np.array([rng.choice([np.nan, -np.inf, np.inf, -0.0, 0.0, -1.0, 2.5]) for _ in range(V)], np.float32)
        assert O.top_k(z, K) == _brute_topk_nan(z, K)
    Z = np.array([[np.nan, 1.0, np.nan, -np.inf], [2.0, 2.0, 1.0, 0.0]], np.float32)
    assert O.top_k_rows(Z, 3).tolist() == [[1, 3, -1], [0, 1, 2]]
    # a prefill row with fewer than K_pre orderable values adds only those
    assert O.stream_init([5], np.array([[np.nan, 3.0, np.nan, np.nan]], np.float32), 2) == [5, 1]


# ---------------------------------------------------------------------------
# Stream init against brute force
# ---------------------------------------------------------------------------
def test_stream_init_brute_force():
    rng = random.Random(7)
    for _ in range(50):
        V = rng.randint(2, 30)
        L = rng.randint(1, 12)
        K = rng.randint(0, 4)
        prompt = [rng.randrange(V) for _ in range(L)]
        Z = np.array([[rng.choice([0.0, 1.0, 2.0, 5.0]) for _ in range(V)] for _ in range(L)], np.float32)
        want = list(prompt)
        emitted = []
        for i in range(L):
            for x in _brute_topk(Z[i], K):
                if x not in emitted:
                    emitted.append(x)
        want += emitted
        # row_chunk=3 also exercises the chunked ranking
        assert O.stream_init(prompt, Z, K, row_chunk=3) == want


# ---------------------------------------------------------------------------
# Window against an independent incremental implementation
# ---------------------------------------------------------------------------
class _CountWindow:
    """Occurrence counts over the last W entries, updated one entry at a time."""

    def __init__(self, W):
        self.W, self.buf, self.count = W, [], {}

    def push(self, x):
        self.buf.append(x)
        self.count[x] = self.count.get(x, 0) + 1
        if len(self.buf) > self.W:
            y = self.buf[len(self.buf) - self.W - 1]
            self.count[y] -= 1
            if self.count[y] == 0:
                del self.count[y]

    def active(self):
        return sorted(self.count)


def test_window_matches_incremental_counts():
    rng = random.Random(99)
    for _ in range(40):
        V = rng.randint(1, 50)
        W = rng.randint(1, 30)
        win = _CountWindow(W)
        S = []
        for _ in range(rng.randint(0, 120)):
            x = rng.randrange(V)
            S.append(x)
            win.push(x)
            I = O.active_vocab(S, W)
            assert I.tolist() == win.active()


def test_window_invariants_random_streams():
    rng = random.Random(3)
    for _ in range(60):
        V = rng.randint(1, 300)
        W = rng.randint(1, 64)
        S = [rng.randrange(V) for _ in range(rng.randint(1, 200))]
        I = O.active_vocab(S, W)
        bm = O.bitmap_words(I, V)
        assert len(I) <= W
        assert all(I[i] < I[i + 1] for i in range(len(I) - 1))
        assert int(sum(bin(int(w)).count("1") for w in bm)) == len(I)
        start = max(0, len(S) - W)
        last = {x: p for p, x in enumerate(S)}
        for x in I.tolist():
            assert last[x] >= start  # most recent occurrence inside the window
        for x in S[start:]:
            assert x in set(I.tolist())
        if V % 32:
            assert int(bm[-1]) >> (V % 32) == 0  # padding bits stay clear


def test_window_special_cases():
    S = [5, 1, 5, 9, 2, 9]
    assert O.active_vocab(S, 100).tolist() == sorted(set(S))  # W >= |S|: everything seen
    assert O.active_vocab(S, 1).tolist() == [9]  # W = 1: the last entry
    S2 = O.stream_append(S, [], None, 0)  # empty tree, no verify candidates
    assert S2 == S and O.active_vocab(S2, 3).tolist() == O.active_vocab(S, 3).tolist()
    with pytest.raises(ValueError):
        O.active_vocab(S, 0)


def test_draft_candidates_first_occurrence():
    assert O.draft_candidates([4, 4, 2, 9, 2, 4, 1]) == [4, 2, 9, 1]
    assert O.draft_candidates([]) == []


# ---------------------------------------------------------------------------
# bf16 decoding, gather, projection, top-k remap
# ---------------------------------------------------------------------------
def test_bf16_values():
    bits = np.array([0x3F80, 0xC000, 0x3D80, 0x0001, 0x7F7F, 0x8000, 0x4049], np.uint16)
    want = [1.0, -2.0, 0.0625, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, -0.0, 3.140625]
    got = O.bf16_to_f64(bits).tolist()
    assert got == want
    assert np.signbit(O.bf16_to_f64(np.array([0x8000], np.uint16)))[0]


# bf16 bit patterns of small exact values, written out by hand.
_BF16 = {-2: 0xC000, -1: 0xBF80, 0: 0x0000, 1: 0x3F80, 2: 0x4000}
_W16 = {-1: 0xBD80, 0: 0x0000, 1: 0x3D80}  # (-1, 0, 1) * 2**-4


def _exact_case(seed, n, m, H, V=None):
    rng = random.Random(seed)
    hid_i = [[rng.randint(-2, 2) for _ in range(H)] for _ in range(n)]
    V = V or m
    w_i = [[rng.randint(-1, 1) for _ in range(H)] for _ in range(V)]
    hid = np.array([[_BF16[v] for v in row] for row in hid_i], np.uint16)
    W = np.array([[_W16[v] for v in row] for row in w_i], np.uint16)
    return hid_i, w_i, hid, W


def test_projection_exact_integer_case():
    hid_i, w_i, hid, W = _exact_case(11, n=5, m=7, H=96)
    logits = O.project(hid, W)
    for r in range(5):
        for j in range(7):
            want = sum(a * b for a, b in zip(hid_i[r], w_i[j])) / 16.0
            assert logits[r, j] == np.float32(want)
    assert logits.shape == (5, 7) and logits.dtype == np.float32


def test_projection_not_transposed_and_single_rounding():
    # one hidden row against two distinct weight rows; an operand swap changes shapes/values
    hid = np.array([[0x3F80, 0x4000, 0x0000]], np.uint16)  # (1, 2, 0)
    W = np.array([[0x3F80, 0x0000, 0x4040], [0x0000, 0xBF80, 0x3F80]], np.uint16)  # (1,0,3), (0,-1,1)
    assert O.project(hid, W).tolist() == [[1.0, -2.0]]
    # fp64 accumulate then one fp32 rounding: 1 + 2^-30 - 1 would lose the small term in fp32
    a = np.array([[0x3F80, 0x3F80, 0x3F80]], np.uint16)  # (1, 1, 1)
    b = np.array([[0x3F80, 0x3080, 0xBF80]], np.uint16)  # (1, 2^-30, -1)
    assert O.project(a, b)[0, 0] == np.float32(2.0 ** -30)


def test_gather_is_row_copy():
    rng = np.random.default_rng(0)
    W = rng.integers(0, 2 ** 16, size=(50, 24), dtype=np.uint16)
    I = np.array([0, 3, 17, 49], np.int32)
    P = O.gather_rows(W, I)
    for j, i in enumerate(I):
        assert P[j].tobytes() == W[i].tobytes()
    assert O.gather_rows(W, np.zeros(0, np.int32)).shape == (0, 24)


def test_subhead_logits_equal_full_vocab_logits_at_I():
    _, _, hid, W = _exact_case(21, n=4, m=0, H=64, V=60)
    I = np.array([1, 5, 6, 30, 59], np.int32)
    full = O.dense_logits(hid, W)
    packed, sub, _, _ = O.sub_head_step(hid, W, I, 3)
    assert np.array_equal(sub, full[:, I])


def test_topk_remap_is_masked_full_vocab_argmax():
    rng = np.random.default_rng(8)
    V, H = 90, 32
    W = rng.integers(0, 2 ** 16, size=(V, H), dtype=np.uint16)
    W = np.where((W & 0x7F80) == 0x7F80, np.uint16(0x3F80), W)  # no inf/nan patterns
    W = (W & np.uint16(0x87FF)) | np.uint16(0x3800)  # modest exponents
    hid = np.array([[_BF16[int(v)] for v in row] for row in rng.integers(-2, 3, size=(6, H))], np.uint16)
    I = np.array(sorted(rng.choice(V, size=25, replace=False)), np.int32)
    full = O.dense_logits(hid, W)
    _, _, ids, vals = O.sub_head_step(hid, W, I, 10)
    member = set(I.tolist())
    for r in range(6):
        brute = sorted((i for i in range(V) if i in member), key=lambda i: (-float(full[r, i]), i))[:10]
        assert ids[r].tolist() == brute
        assert vals[r].tolist() == [float(full[r, i]) for i in brute]


def test_topk_remap_pads_short_rows():
    logits = np.array([[0.5, 2.0], [1.0, 1.0]], np.float32)
    ids, vals = O.topk_remap(logits, np.array([7, 3], np.int32), 4)
    assert ids.tolist() == [[3, 7, -1, -1], [7, 3, -1, -1]]
    assert vals[0, :2].tolist() == [2.0, 0.5] and np.all(np.isneginf(vals[:, 2:]))
    ids0, vals0 = O.topk_remap(np.zeros((2, 0), np.float32), np.zeros(0, np.int32), 3)
    assert (ids0 == -1).all() and np.isneginf(vals0).all()


def test_topk_remap_pads_rows_with_few_orderable_values():
    # NaN never ranks: a row with fewer than k non-NaN logits ends in (-1, -inf)
    # padding, whatever its width; infinities rank like any value
    logits = np.array([[np.nan, 2.0, np.nan, np.inf, np.nan, -np.inf],
                       [np.nan] * 6], dtype=np.float32)
    I = np.array([10, 11, 12, 13, 14, 15])
    ids, vals = O.topk_remap(logits, I, 4)
    assert ids.tolist() == [[13, 11, 15, -1], [-1, -1, -1, -1]]
    assert vals[0, :3].tolist() == [np.inf, 2.0, -np.inf] and np.isneginf(vals[0, 3]) and np.all(np.isneginf(vals[1]))
