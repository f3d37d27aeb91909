"""Seeded synthetic inputs for the MaxSim rerank of one query against packed documents.

Layout follows the vLLM page "flash_maxsim_rerank" (flash_maxsim_rerank_direct): one
query ``q [lq, d]`` fp16 and a packed ``[total_tokens, d]`` fp16 tensor that holds every
request's tokens, the documents being ``(offset, length)`` pairs into it, scattered and
not contiguous. Like the rest of ``workloads`` this module only draws random numbers and
lays out rows; it computes no similarity, no maximum and no sum.

Recipe (seeded; ``numpy.random.SeedSequence(seed).spawn(3)`` gives independent streams
for values, lengths and placement):

* values: ``"normal"`` draws N(0,1)/sqrt(d) (about unit-norm embeddings, as a late-
  interaction encoder emits), ``"int"`` draws integers in {-3..3} so that every dot
  product and sum is exact in fp32;
* lengths: uniform integers in ``[len_lo, len_hi]``, after any ``fixed_lengths``;
* placement: the documents go into the tensor in a random order, each after a gap of
  uniform ``[0, gap_hi]`` rows of "other" tokens; the gap rows (and rows past the last
  document) are poisoned with ``60 * sign(q[0])``, which would win query row 0's maximum
  in any document that read them;
* ``extra_docs`` adds documents that overlap others, start before row 0 or run past the
  last row (rows outside the tensor read as zero vectors).
"""

from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass
class MaxsimWorkload:
    name: str
    q: np.ndarray        # fp16 [lq, d]
    docs: np.ndarray     # fp16 [total_tokens, d]
    offsets: np.ndarray  # int32 [B]
    lengths: np.ndarray  # int32 [B]

    @property
    def num_docs(self) -> int:
        return int(self.offsets.size)

    @property
    def doc_rows(self) -> int:
        """Rows the documents name (with repeats), the unit of the throughput metric."""
        return int(np.maximum(self.lengths, 0).sum())


def build_maxsim(*, name: str, lq: int, d: int, num_docs: int, len_lo: int, len_hi: int, seed: int,
                 gap_hi: int = 32, values: str = "normal", fixed_lengths=(), extra_docs: bool = False
                 ) -> MaxsimWorkload:
    s_val, s_len, s_place = (np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(3))
    fixed = np.asarray(fixed_lengths, dtype=np.int64)
    n_rand = max(0, num_docs - fixed.size)
    lengths = np.concatenate([fixed, s_len.integers(len_lo, len_hi + 1, size=n_rand)])[:num_docs]
    if values == "int":
        q = s_val.integers(-3, 4, size=(lq, d)).astype(np.float16)
    else:
        q = (s_val.standard_normal((lq, d)) / np.sqrt(d)).astype(np.float16)
    order = s_place.permutation(num_docs)
    gaps = s_place.integers(0, gap_hi + 1, size=num_docs)
    total = int(gaps.sum() + np.maximum(lengths, 0).sum()) + gap_hi + 1
    poison = (60.0 * np.sign(q[0].astype(np.float32) + 1e-3)).astype(np.float16) if lq else np.zeros(d, np.float16)
    docs = np.empty((total, d), dtype=np.float16)
    docs[:] = poison
    offsets = np.zeros(num_docs, dtype=np.int64)
    cur = 0
    for i in order:
        cur += int(gaps[i])
        n = max(int(lengths[i]), 0)
        offsets[i] = cur
        if values == "int":
            docs[cur:cur + n] = s_val.integers(-3, 4, size=(n, d)).astype(np.float16)
        else:
            docs[cur:cur + n] = (s_val.standard_normal((n, d)) / np.sqrt(d)).astype(np.float16)
        cur += n
    if extra_docs and num_docs > 0:
        # overlapping an existing document, before row 0, past the end, and a 1-row one
        big = int(np.argmax(lengths))
        extra_off = [offsets[big] + max(int(lengths[big]) // 3, 0), -5, total - 7, offsets[big]]
        extra_len = [max(int(lengths[big]) // 2, 1), 9, 40, 1]
        offsets = np.concatenate([offsets, extra_off])
        lengths = np.concatenate([lengths, extra_len])
    return MaxsimWorkload(name=name, q=q, docs=docs, offsets=offsets.astype(np.int32),
                          lengths=lengths.astype(np.int32))


# Named configurations: the small ragged case the oracle checks whole, and the rerank
# batch timed by the benchmark (ColBERT-style 32 x 128 query, 4096 candidate documents of
# 1..512 rows, about 1.05 M rows = 270 MB of fp16, above the 129 MB L2).
MAXSIM_CONFIGS = {
    "maxsim_small": dict(lq=32, d=128, num_docs=40, len_lo=0, len_hi=300, gap_hi=40,
                         fixed_lengths=(0, 1, 2, 31, 32, 33, 64, 65, 127, 128, 129, 513, -3), extra_docs=True),
    "maxsim_rerank4k": dict(lq=32, d=128, num_docs=4096, len_lo=1, len_hi=512, gap_hi=64),
}
MAXSIM_SEEDS = {"maxsim_small": 2001, "maxsim_rerank4k": 2002}


def make_maxsim(name: str, seed: int | None = None, **overrides) -> MaxsimWorkload:
    cfg = dict(MAXSIM_CONFIGS[name], **overrides)
    return build_maxsim(name=name, seed=MAXSIM_SEEDS[name] if seed is None else seed, **cfg)
