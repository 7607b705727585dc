"""Plain CPU restatement of the dynamic-vocabulary draft LM head.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.

Sources (the paper appears on two pages, once as NanoSpec and once as
MicroSpec; section numbers are MicroSpec's, which keeps its headings):

* [Eq. 1]   MicroSpec §3.1 "Preliminaries and Problem Formulation", Eq. 1:
            z_t = W_head h_t, W_head in R^{V x d}.
* [T_K]     MicroSpec §3.2 "Candidate Stream Initialization": T_K(z) is the
            set of indices of the K largest values of z.
* [S_init]  MicroSpec §3.2, stream-initialisation equation:
            S_init = (x_1..x_L) (+) tuple(U_{i=1..L} T_Kpre(z_i)).
* [C_draft] MicroSpec §3.2 "Dynamic Stream Update", item 1: all unique token
            ids anywhere in the draft tree, accepted or not.
* [C_ver]   MicroSpec §3.2, item 2: C_ver = T_Kver(z_verify).
* [S_new]   MicroSpec §3.2, stream-update equation:
            S_new = S_old (+) tuple(C_draft) (+) tuple(C_ver).
* [I_t]     MicroSpec §3.2 "Vocabulary Construction via Sliding Window":
            I_{t+1} = Unique(Suffix(S_new, W_max)); NanoSpec's same paragraph
            adds that a token whose most recent occurrence falls outside the
            window is discarded.
* [gather]  MicroSpec §3.3 "Avoiding Sparse Computation via Asynchronous
            Gathering": rows W_head[I_t, :] packed contiguously, then a dense
            product.
* [bitmap]  MicroSpec §3.3 "Eliminating Overhead via GPU-Resident State
            Management": the active window kept as bitmaps.
* [slots]   NanoSpec, "Avoiding Sparse Computation via Asynchronous
            Gathering": the weights of newly active tokens are gathered into
            the pre-allocated contiguous buffer.

Readings where the pages are silent (each also listed in the design notes):

1. tuple() order: first occurrence.  S_init's union is walked position-major
   (i = 1..L), rank-minor (largest logit first); C_draft keeps node order;
   C_ver keeps rank order.
2. Append everything the formal definition appends, so a re-seen id refreshes
   its recency (duplicates between C_draft and C_ver are kept too).
3. Ties in T_K: larger value first, then the smaller id.  Comparisons are made
   on the fp32 inputs exactly (fp64 holds every fp32 value); -0.0 ties +0.0.
   NaN never ranks; -inf and +inf are ordered like any other value.  A row
   with fewer than K orderable (non-NaN) values gives fewer than K picks.
4. Unique() yields ascending ids.
5. Suffix of a stream shorter than W_max is the whole stream.
6. Prompt ids are kept verbatim (with repeats); only the Top-K union is
   deduplicated.
7. Token ids are 0-based.
8. Logits of the projection: exact products of bf16 inputs summed in fp64,
   rounded once to fp32.
9. Top-k of a row with fewer than k active columns is padded with id -1 and
   value -inf.
10. Slot-stable buffer (the incremental reading of [gather]: only the rows of
   newly active tokens are gathered).  The pages fix no slot rule; here a
   slot whose id left I_t is freed, and the ids of I_t that hold no slot take
   the free slots in ascending id order, lowest slot first.  The first update
   after the stream is initialised therefore lays I_1 out ascending, the same
   layout as the full repack.
11. Batched shared gather (several sequences' sub-heads from one packed
   buffer): the buffer holds the union U of the sequences' I_t, ascending;
   each sequence projects through all of it and ranks only its own columns,
   so its top-k is the one its own I_t gives.

"""

from __future__ import annotations

from typing import Iterable, List, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# bf16 values
# ---------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as fp64.

    A bf16 number is the upper half of an fp32 number, so the pattern shifted
    left by 16 is that fp32 number, which fp64 holds exactly.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Top-K operator [T_K]
# ---------------------------------------------------------------------------
def top_k_rows(Z, K: int) -> np.ndarray:
    """T_K of every row of Z, as ordered index lists (int64 [rows, min(K, V)]).

    Pick r (r = 0..K-1) is the largest value not yet picked; among equal
    values the smallest index wins.  This is exactly the first K entries of a
    stable descending sort of the row's orderable (non-NaN) values.  Rows of
    finite values take K rounds of argmax (numpy's argmax returns the first
    maximum; picked entries are set to -inf, which no finite input reaches);
    rows holding NaN or an infinity are sorted.  A row with fewer than K
    orderable values is padded with -1.
    """
    Z = np.asarray(Z, dtype=np.float32)
    if Z.ndim != 2:
        raise ValueError("top_k_rows expects a 2-D array")
    n, V = Z.shape
    K = min(int(K), V)
    out = np.full((n, max(K, 0)), -1, dtype=np.int64)
    if K <= 0 or n == 0:
        return out
    finite = np.all(np.isfinite(Z), axis=1)
    rows = np.flatnonzero(finite)
    if len(rows):
        work = Z[rows].astype(np.float64)
        sel = np.arange(len(rows))
        for r in range(K):
            j = np.argmax(work, axis=1)
            out[rows, r] = j
            work[sel, j] = -np.inf
    for i in np.flatnonzero(~finite):
        z = Z[i].astype(np.float64)
        ids = np.flatnonzero(~np.isnan(z))
        order = ids[np.lexsort((ids, -z[ids]))]  # value descending, then id ascending
        take = order[:K]
        out[i, :len(take)] = take
    return out


def top_k(z, K: int) -> List[int]:
    """T_K(z) of one logit vector, best first (fewer than K ids when the
    vector has fewer than K orderable values)."""
    z = np.asarray(z, dtype=np.float32).reshape(1, -1)
    return [int(x) for x in top_k_rows(z, K)[0] if x >= 0]


# ---------------------------------------------------------------------------
# Candidate stream [S_init], [C_draft], [C_ver], [S_new]
# ---------------------------------------------------------------------------
def stream_init(prompt: Sequence[int], prefill_logits, K_pre: int, row_chunk: int = 256) -> List[int]:
    """S_init = prompt (+) tuple(union of T_Kpre(z_i), i = 1..L).

    The union is read out in first-occurrence order, position-major and
    rank-minor.  ``prefill_logits`` is [L, V]; rows are ranked ``row_chunk``
    at a time only to bound memory (each row's ranking is independent).
    """
    S = [int(x) for x in prompt]
    L = len(S)
    if K_pre <= 0 or L == 0:
        return S
    Z = prefill_logits
    if Z.shape[0] != L:
        raise ValueError("need one prefill logit row per prompt position")
    seen = set()
    for r0 in range(0, L, row_chunk):
        T = top_k_rows(Z[r0:r0 + row_chunk], K_pre)
        for i in range(T.shape[0]):
            for x in T[i]:
                x = int(x)
                if x >= 0 and x not in seen:  # -1 pads a row with fewer than K_pre orderable values
                    seen.add(x)
                    S.append(x)
    return S


def draft_candidates(tree_ids: Iterable[int]) -> List[int]:
    """C_draft: the distinct ids of the draft tree, in first-occurrence node order."""
    seen = set()
    out = []
    for x in tree_ids:
        x = int(x)
        if x not in seen:
            seen.add(x)
            out.append(x)
    return out


def stream_append(S: Sequence[int], tree_ids, z_verify, K_ver: int) -> List[int]:
    """S_new = S_old (+) tuple(C_draft) (+) tuple(C_ver), C_ver = T_Kver(z_verify)."""
    c_draft = draft_candidates(tree_ids)
    c_ver = top_k(z_verify, K_ver) if K_ver > 0 else []
    return list(S) + c_draft + c_ver


# ---------------------------------------------------------------------------
# Sliding-window active vocabulary [I_t], [bitmap]
# ---------------------------------------------------------------------------
def active_vocab(S: Sequence[int], W_max: int) -> np.ndarray:
    """I = Unique(Suffix(S, W_max)), ascending (int32)."""
    if W_max <= 0:
        raise ValueError("W_max must be positive")
    suffix = list(S)[-W_max:]
    return np.array(sorted(set(suffix)), dtype=np.int32)


def bitmap_words(I, V: int) -> np.ndarray:
    """Membership bitmap of I over ids 0..V-1: bit (i % 32) of word i // 32."""
    words = np.zeros((V + 31) // 32, dtype=np.uint32)
    for i in np.asarray(I, dtype=np.int64).tolist():
        if not 0 <= i < V:
            raise ValueError("id out of range")
        words[i >> 5] |= np.uint32(1 << (i & 31))
    return words


# ---------------------------------------------------------------------------
# Sub-head [gather], projection [Eq. 1] and top-k
# ---------------------------------------------------------------------------
def gather_rows(W_bits, I) -> np.ndarray:
    """packed[j, :] = W_head[I[j], :] (bf16 bit patterns, byte copy)."""
    W_bits = np.asarray(W_bits, dtype=np.uint16)
    return W_bits[np.asarray(I, dtype=np.int64)].copy()


def project(hid_bits, rows_bits) -> np.ndarray:
    """logits[r, j] = sum_h hid[r, h] * rows[j, h]  (Eq. 1 restricted to the given rows).

    bf16 inputs are exact in fp64; the sum is an fp64 matrix product, rounded
    once to fp32.  Returns fp32 [n, m].
    """
    h = bf16_to_f64(hid_bits)
    w = bf16_to_f64(rows_bits)
    if h.ndim != 2 or w.ndim != 2 or h.shape[1] != w.shape[1]:
        raise ValueError("shape mismatch")
    return (h @ w.T).astype(np.float32)


def dense_logits(hid_bits, W_bits) -> np.ndarray:
    """Full-vocabulary logits z = W_head h for every hidden row (fp32 [n, V])."""
    return project(hid_bits, W_bits)


def topk_remap(logits, I, k: int):
    """Per row, the top-k columns of ``logits`` mapped to global ids through I.

    Returns (ids int32 [n, k], vals fp32 [n, k]); rows with fewer than k
    orderable (non-NaN) columns are padded with (-1, -inf).
    """
    logits = np.asarray(logits, dtype=np.float32)
    I = np.asarray(I, dtype=np.int64)
    n, m = logits.shape
    ids = np.full((n, k), -1, dtype=np.int32)
    vals = np.full((n, k), -np.inf, dtype=np.float32)
    kk = min(k, m)
    if kk > 0 and n > 0:
        T = top_k_rows(logits, kk)
        for r in range(n):
            t = T[r][T[r] >= 0]
            ids[r, :len(t)] = I[t]
            vals[r, :len(t)] = logits[r, t]
    return ids, vals


def sub_head_step(hid_bits, W_bits, I, k: int):
    """Gather, project and top-k for one step: (packed, logits, ids, vals)."""
    packed = gather_rows(W_bits, I)
    logits = project(hid_bits, packed)
    ids, vals = topk_remap(logits, I, k)
    return packed, logits, ids, vals


# ---------------------------------------------------------------------------
# Slot-stable packed buffer [slots] (reading 10)
# ---------------------------------------------------------------------------
def slot_update(slot_id, I):
    """One update of the slot table to the active set I.

    ``slot_id`` has one entry per buffer slot (W_max of them): the id held,
    or -1 for a free slot.  Returns (new table, new_pairs): every slot whose
    id is not in I is freed; then the ids of I that hold no slot, ascending,
    take the free slots, lowest slot first.  ``new_pairs`` lists the
    (slot, id) assignments made, in that order; they are the rows to gather.
    """
    table = [int(x) for x in slot_id]
    active = set(int(x) for x in I)
    if len(active) > len(table):
        raise ValueError("more active ids than slots")
    for sl, x in enumerate(table):
        if x >= 0 and x not in active:
            table[sl] = -1
    held = set(x for x in table if x >= 0)
    new_ids = sorted(active - held)
    free = [sl for sl, x in enumerate(table) if x < 0]
    pairs = list(zip(free, new_ids))
    for sl, x in pairs:
        table[sl] = x
    return np.array(table, dtype=np.int32), pairs


def slot_high_water(slot_id) -> int:
    """One past the highest occupied slot (0 for an empty table)."""
    occ = np.flatnonzero(np.asarray(slot_id) >= 0)
    return int(occ[-1]) + 1 if len(occ) else 0


def slot_gather(rows_bits, W_bits, pairs) -> np.ndarray:
    """The buffer after copying W_head[id, :] into slot ``slot`` for every
    (slot, id) in ``pairs``; every other slot keeps its bytes."""
    out = np.array(rows_bits, dtype=np.uint16, copy=True)
    W_bits = np.asarray(W_bits, dtype=np.uint16)
    for sl, x in pairs:
        out[sl] = W_bits[x]
    return out


def slot_project_topk(hid_bits, rows_bits, slot_id, k: int):
    """Projection over the slot buffer and per-row top-k of the occupied slots.

    Returns (logits fp32 [n, hw], ids, vals): logits[r, s] = Eq. 1 over slot
    s's row for s < hw (free slots included, unranked); the top-k ranks only
    occupied slots, maps them to the ids they hold and orders by value, then
    the smaller id, exactly as the full repack does (its columns are the ids
    in ascending order).
    """
    slot_id = np.asarray(slot_id, dtype=np.int64)
    hw = slot_high_water(slot_id)
    logits = project(hid_bits, np.asarray(rows_bits)[:hw])
    occ = np.flatnonzero(slot_id[:hw] >= 0)
    by_id = occ[np.argsort(slot_id[occ], kind="stable")]  # occupied slots, ids ascending
    ids, vals = topk_remap(logits[:, by_id], slot_id[by_id], k)
    return logits, ids, vals


# ---------------------------------------------------------------------------
# Batched shared gather [gather] over several sequences (reading 11)
# ---------------------------------------------------------------------------
def union_vocab(I_list):
    """U = the union of the sequences' active sets, ascending, and the mask
    M[b, j] = (U[j] in I_b) of which columns each sequence may rank."""
    U = np.array(sorted(set(int(x) for I in I_list for x in I)), dtype=np.int32)
    M = np.zeros((len(I_list), len(U)), dtype=bool)
    pos = {int(x): j for j, x in enumerate(U.tolist())}
    for b, I in enumerate(I_list):
        for x in I:
            M[b, pos[int(x)]] = True
    return U, M


def union_sub_head_step(hid_list, W_bits, I_list, k: int):
    """One gather of W_head[U, :] for all sequences, every sequence's hidden
    rows projected through it, and each sequence's top-k over its own columns
    only.  Returns (U, M, packed [|U| x H], logits per sequence [n_b x |U|],
    ids, vals per sequence)."""
    U, M = union_vocab(I_list)
    packed = gather_rows(W_bits, U)
    logits, ids, vals = [], [], []
    for b, hid in enumerate(hid_list):
        z = project(hid, packed)
        cols = np.flatnonzero(M[b])  # ascending, so ids ascend with the column
        i_b, v_b = topk_remap(z[:, cols], U[cols], k)
        logits.append(z)
        ids.append(i_b)
        vals.append(v_b)
    return U, M, packed, logits, ids, vals


class OracleSlots:
    """The slot table and buffer of one sequence."""

    def __init__(self, W_max: int, H: int):
        self.slot_id = np.full(W_max, -1, dtype=np.int32)
        self.rows = np.zeros((W_max, H), dtype=np.uint16)

    def update(self, I, W_bits):
        self.slot_id, pairs = slot_update(self.slot_id, I)
        self.rows = slot_gather(self.rows, W_bits, pairs)
        return pairs

    def project_topk(self, hid_bits, k: int):
        return slot_project_topk(hid_bits, self.rows, self.slot_id, k)


# ---------------------------------------------------------------------------
# Convenience state holder
# ---------------------------------------------------------------------------
class OracleStream:
    """The whole candidate stream of one sequence, kept as a Python list."""

    def __init__(self, V: int, W_max: int, K_pre: int, K_ver: int):
        self.V, self.W_max, self.K_pre, self.K_ver = V, W_max, K_pre, K_ver
        self.S: List[int] = []

    def init(self, prompt, prefill_logits) -> None:
        self.S = stream_init(prompt, prefill_logits, self.K_pre)

    def append(self, tree_ids, verify_block, verify_row: int) -> None:
        z = None if self.K_ver == 0 else np.asarray(verify_block)[verify_row]
        self.S = stream_append(self.S, tree_ids, z, self.K_ver)

    def active(self) -> np.ndarray:
        return active_vocab(self.S, self.W_max)

    def bitmap(self) -> np.ndarray:
        return bitmap_words(self.active(), self.V)
