"""Seeded synthetic workloads shaped like the draft LM heads the method targets.

Every random number comes from numpy's PCG64 bit generator, keyed by a
``SeedSequence([seed, seq, tag, index])`` and read only through
``random_raw`` (raw 64-bit words, whose stream numpy keeps stable across
versions and platforms).  All values are derived from those words with integer
operations and single, exactly specified fp32 roundings, so a given key always
yields the same bytes.

Distributions (one recipe for every workload):

* ``Zipf(s)`` over ranks ``1..V``: inverse CDF of ``r**-s`` built once in
  fp64; rank ``r`` is token id ``r-1``, so low ids are the frequent ones (the
  "first 32768 ids" are a frequency-ranked static sub-vocabulary).
* random fp32 logits: ``(top 24 bits of a raw word) * 2**-20 - 8``, exact fp32
  values in ``[-8, 8)``.
* ``N(0, sigma)`` in bf16: Irwin-Hall sum of the four 16-bit fields of one raw
  word, centred, times ``sigma / 37837.2`` in one fp32 multiply (37837.2 is the
  standard deviation of that sum), then rounded to bf16 to nearest-even.
* self-copy prompts: with probability ``p`` a position copies a uniformly
  chosen earlier prompt id, otherwise it draws Zipf.
* draft trees: each node, with probability ``f``, copies a uniform entry of
  the last ``R`` ids of the generator's own history (prompt followed by all
  earlier tree ids), otherwise draws Zipf.

Token ids are 0-based (the papers number the vocabulary ``1..V``).
"""

from __future__ import annotations

import dataclasses
import os
from dataclasses import dataclass
from functools import lru_cache
from typing import Optional

import numpy as np

# Stream tags: one independent random stream per kind of input.
TAG_W = 1
TAG_PROMPT = 2
TAG_PREFILL = 3
TAG_TREE = 4
TAG_VERIFY = 5
TAG_VROW = 6
TAG_HIDDEN = 7
TAG_PLEN = 8

W_ROW_CHUNK = 256  # W_head rows drawn per random stream
IRWIN_HALL4_STD = 37837.2  # std of the sum of four uniform 16-bit integers
IRWIN_HALL4_MEAN = 131070  # mean of that sum: 4 * 65535 / 2


def raw_words(seed: int, seq: int, tag: int, index: int, n: int) -> np.ndarray:
    """``n`` raw uint64 words of the stream keyed by (seed, seq, tag, index)."""
    if n == 0:
        return np.zeros(0, dtype=np.uint64)
    bitgen = np.random.PCG64(np.random.SeedSequence([seed, seq, tag, index]))
    return bitgen.random_raw(n)


def unit_f64(raw: np.ndarray) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of each raw word."""
    return (raw >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (rounded & np.uint64(0xFFFF)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16_bits(raw: np.ndarray, sigma: float) -> np.ndarray:
    """Approximate N(0, sigma) samples as bf16 bits, one per raw word."""
    m = np.uint64(0xFFFF)
    s = (raw & m) + ((raw >> np.uint64(16)) & m) + ((raw >> np.uint64(32)) & m) + (raw >> np.uint64(48))
    centred = s.astype(np.int64) - IRWIN_HALL4_MEAN
    x = centred.astype(np.float32) * np.float32(sigma / IRWIN_HALL4_STD)
    return f32_to_bf16_bits(x)


def logits_f32(raw: np.ndarray) -> np.ndarray:
    """Exact fp32 logits in [-8, 8) with a 2**-20 grid."""
    top24 = (raw >> np.uint64(40)).astype(np.float32)
    return top24 * np.float32(2.0 ** -20) - np.float32(8.0)


@lru_cache(maxsize=16)
def zipf_cdf(V: int, s: float) -> np.ndarray:
    """Normalised CDF of Zipf(s) over ranks 1..V (fp64)."""
    w = np.power(np.arange(1, V + 1, dtype=np.float64), -s)
    c = np.cumsum(w)
    return c / c[-1]


def zipf_ids(V: int, s: float, u: np.ndarray) -> np.ndarray:
    """Inverse-CDF Zipf draws; returns 0-based token ids."""
    idx = np.searchsorted(zipf_cdf(V, s), u, side="right")
    return np.minimum(idx, V - 1).astype(np.int32)


@dataclass(frozen=True)
class WorkloadConfig:
    """Shape and recipe of one synthetic workload (all sequences share W_head)."""

    name: str
    V: int
    H: int
    W_max: int
    K_pre: int
    K_ver: int
    prompt_len: int  # fixed prompt length (prompt_len_max > 0 overrides)
    self_copy: float  # probability a prompt position copies an earlier prompt id
    zipf_s: float
    steps: int  # decode steps
    n_tree: int  # draft-tree nodes per step (= hidden rows)
    tree_local: float  # probability a tree node resamples recent history
    tree_recent: int  # how many recent history entries it resamples from
    n_verify: int  # rows of the verify-logits block handed over per step
    k: int = 10  # top-k taken per hidden row
    batch: int = 1  # independent sequences
    prompt_len_min: int = 0  # batched workloads: prompt length ~ U[min, max]
    prompt_len_max: int = 0
    sigma_w: float = 0.02
    seed: int = 0
    W_max_sweep: tuple = ()

    def with_(self, **kw) -> "WorkloadConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    # Toy: V=4096, H=256, W_max=512, 16 steps of a 16-node tree, 16 verify rows.
    "toy_v4096_h256": WorkloadConfig(
        name="toy_v4096_h256", V=4096, H=256, W_max=512, K_pre=3, K_ver=3,
        prompt_len=256, self_copy=0.0, zipf_s=1.1, steps=16, n_tree=16,
        tree_local=0.70, tree_recent=128, n_verify=16),
    # Llama-3-8B-shaped draft head.
    "llama3_8b_v128256_h4096": WorkloadConfig(
        name="llama3_8b_v128256_h4096", V=128256, H=4096, W_max=3072, K_pre=3, K_ver=3,
        prompt_len=1024, self_copy=0.60, zipf_s=1.1, steps=256, n_tree=60,
        tree_local=0.75, tree_recent=512, n_verify=1),
    # Qwen-2.5-7B-shaped draft head.
    "qwen25_7b_v152064_h3584": WorkloadConfig(
        name="qwen25_7b_v152064_h3584", V=152064, H=3584, W_max=3072, K_pre=3, K_ver=3,
        prompt_len=2048, self_copy=0.60, zipf_s=1.05, steps=512, n_tree=60,
        tree_local=0.75, tree_recent=512, n_verify=1),
    # Qwen3-8B-shaped sweep over W_max (default point 3072).
    "qwen3_8b_v151936_h4096": WorkloadConfig(
        name="qwen3_8b_v151936_h4096", V=151936, H=4096, W_max=3072, K_pre=3, K_ver=3,
        prompt_len=4096, self_copy=0.50, zipf_s=1.0, steps=256, n_tree=60,
        tree_local=0.75, tree_recent=512, n_verify=1,
        W_max_sweep=(512, 1024, 2048, 3072, 4096, 8192)),
    # Batched serving: 16 independent Llama-3-shaped sequences.
    "batched16_v128256_h4096": WorkloadConfig(
        name="batched16_v128256_h4096", V=128256, H=4096, W_max=3072, K_pre=3, K_ver=3,
        prompt_len=0, prompt_len_min=512, prompt_len_max=4096, self_copy=0.60, zipf_s=1.1,
        steps=128, n_tree=60, tree_local=0.75, tree_recent=512, n_verify=1, batch=16),
}


def get_config(name: str) -> WorkloadConfig:
    return CONFIGS[name]


class Workload:
    """Lazily generated inputs of one WorkloadConfig.

    Arrays are numpy host arrays: token ids int32, logits fp32, bf16 tensors as
    uint16 bit patterns.
    """

    def __init__(self, cfg: WorkloadConfig):
        self.cfg = cfg
        self._w: Optional[np.ndarray] = None
        self._prompts: dict = {}
        self._trees: dict = {}

    # -- model weights -------------------------------------------------------
    def w_head_rows(self, r0: int, r1: int) -> np.ndarray:
        """Rows [r0, r1) of W_head (bf16 bits, [r1-r0, H])."""
        c = self.cfg
        out = np.empty((r1 - r0, c.H), dtype=np.uint16)
        ch0, ch1 = r0 // W_ROW_CHUNK, (r1 - 1) // W_ROW_CHUNK
        for ch in range(ch0, ch1 + 1):
            a = ch * W_ROW_CHUNK
            b = min(a + W_ROW_CHUNK, c.V)
            block = normal_bf16_bits(raw_words(c.seed, 0, TAG_W, ch, (b - a) * c.H), c.sigma_w)
            block = block.reshape(b - a, c.H)
            lo, hi = max(a, r0), min(b, r1)
            out[lo - r0:hi - r0] = block[lo - a:hi - a]
        return out

    def w_head(self) -> np.ndarray:
        """The whole LM head W_head [V, H] (bf16 bits), generated once.

        Row chunks are independent streams, so they are drawn in parallel
        threads (numpy releases the GIL); the bytes do not depend on the
        thread count."""
        if self._w is None:
            from concurrent.futures import ThreadPoolExecutor

            c = self.cfg
            out = np.empty((c.V, c.H), dtype=np.uint16)
            span = 16 * W_ROW_CHUNK

            def fill(r0):
                r1 = min(r0 + span, c.V)
                out[r0:r1] = self.w_head_rows(r0, r1)

            workers = max(1, min(16, os.cpu_count() or 1))
            with ThreadPoolExecutor(max_workers=workers) as ex:
                list(ex.map(fill, range(0, c.V, span)))
            self._w = out
        return self._w

    # -- prompt and prefill --------------------------------------------------
    def prompt_len(self, seq: int = 0) -> int:
        c = self.cfg
        if c.prompt_len_max > 0:
            span = c.prompt_len_max - c.prompt_len_min + 1
            u = unit_f64(raw_words(c.seed, seq, TAG_PLEN, 0, 1))[0]
            return c.prompt_len_min + int(u * span)
        return c.prompt_len

    def prompt(self, seq: int = 0) -> np.ndarray:
        if seq not in self._prompts:
            c = self.cfg
            L = self.prompt_len(seq)
            raw = raw_words(c.seed, seq, TAG_PROMPT, 0, 3 * L)
            u_mode, u_pick = unit_f64(raw[0::3]), unit_f64(raw[1::3])
            z = zipf_ids(c.V, c.zipf_s, unit_f64(raw[2::3]))
            p = np.empty(L, dtype=np.int32)
            for i in range(L):
                if i > 0 and u_mode[i] < c.self_copy:
                    p[i] = p[int(u_pick[i] * i)]
                else:
                    p[i] = z[i]
            self._prompts[seq] = p
        return self._prompts[seq]

    def prefill_logits(self, seq: int = 0, r0: int = 0, r1: Optional[int] = None) -> np.ndarray:
        """Rows [r0, r1) of the target's prefill logits Z_{1:L} (fp32 [rows, V])."""
        c = self.cfg
        L = self.prompt_len(seq)
        r1 = L if r1 is None else r1
        out = np.empty((r1 - r0, c.V), dtype=np.float32)
        for i in range(r0, r1):
            out[i - r0] = logits_f32(raw_words(c.seed, seq, TAG_PREFILL, i, c.V))
        return out

    # -- decode steps --------------------------------------------------------
    def trees(self, seq: int = 0) -> np.ndarray:
        """Draft-tree token ids of every step, int32 [steps, n_tree]."""
        if seq not in self._trees:
            c = self.cfg
            hist = list(self.prompt(seq).tolist())
            out = np.empty((c.steps, c.n_tree), dtype=np.int32)
            for t in range(c.steps):
                raw = raw_words(c.seed, seq, TAG_TREE, t, 3 * c.n_tree)
                u_mode, u_pick = unit_f64(raw[0::3]), unit_f64(raw[1::3])
                z = zipf_ids(c.V, c.zipf_s, unit_f64(raw[2::3]))
                for i in range(c.n_tree):
                    if hist and u_mode[i] < c.tree_local:
                        win = min(c.tree_recent, len(hist))
                        out[t, i] = hist[len(hist) - win + int(u_pick[i] * win)]
                    else:
                        out[t, i] = z[i]
                hist.extend(out[t].tolist())
            self._trees[seq] = out
        return self._trees[seq]

    def verify_logits(self, seq: int, step: int) -> np.ndarray:
        """The verify-logits block of one step, fp32 [n_verify, V]."""
        c = self.cfg
        return logits_f32(raw_words(c.seed, seq, TAG_VERIFY, step, c.n_verify * c.V)).reshape(
            c.n_verify, c.V)

    def verify_row(self, seq: int, step: int) -> int:
        """Row of the verify block that holds the validated branch's logits."""
        c = self.cfg
        if c.n_verify == 1:
            return 0
        u = unit_f64(raw_words(c.seed, seq, TAG_VROW, step, 1))[0]
        return int(u * c.n_verify)

    def hiddens(self, seq: int, step: int) -> np.ndarray:
        """Draft hidden states of one step, bf16 bits [n_tree, H], ~N(0, 1)."""
        c = self.cfg
        return normal_bf16_bits(raw_words(c.seed, seq, TAG_HIDDEN, step, c.n_tree * c.H), 1.0).reshape(
            c.n_tree, c.H)
