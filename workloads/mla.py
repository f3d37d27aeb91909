"""Seeded synthetic inputs for sparse MLA decode attention over selected KV slots.

Layout follows the vLLM page "flashinfer_mla_sparse_sm90" (_SM90State): per decode row a
query of `heads` heads, each a latent part q_nope of kv_lora_rank (dc) dims and a rotary
part q_pe of qk_rope_head_dim (dr, 0 or 64) dims, in bf16; a KV cache of one row per token
slot holding the latent ckv (dc) and the rotary key kpe (dr) side by side (page size 1, so
the selected slots are the page table); per row the selection's slots (ascending, then a
-1 tail) and the exact kv_len of _kv_lens_host (ctx if ctx <= topk else topk + ctx % kpool).
Like the rest of ``workloads`` this module draws random numbers and lays out tables only;
it computes no attention.

Recipe (seeded; ``numpy.random.SeedSequence(seed).spawn(3)``: values, slots, holes):
* bf16 values as bit patterns (uint16): N(0,1) samples truncated to their top 16 bits, scaled
  by 1/sqrt(dc) for q_nope and q_pe; ckv and kpe rows N(0,1);
* each row's kv_len entries are distinct slots drawn uniformly from [0, num_slots), sorted
  ascending, then -1 up to `width`; with `holes`, about 1 % of the entries inside kv_len are
  -1 (an out-of-bounds block in the selection) and a few name a slot past num_slots.
"""

from __future__ import annotations

import dataclasses

import numpy as np


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@dataclasses.dataclass
class MlaWorkload:
    name: str
    q_nope: np.ndarray   # bf16 bits [rows, heads, dc]
    q_pe: np.ndarray     # bf16 bits [rows, heads, dr]
    cache: np.ndarray    # bf16 bits [num_slots, dc + dr]: ckv then kpe per slot
    slots: np.ndarray    # int32 [rows, width]
    kv_len: np.ndarray   # int32 [rows]
    sm_scale: float

    @property
    def dc(self) -> int:
        return int(self.q_nope.shape[2])

    @property
    def dr(self) -> int:
        return int(self.q_pe.shape[2])

    @property
    def ckv(self) -> np.ndarray:
        return self.cache[:, :self.dc]

    @property
    def kpe(self) -> np.ndarray:
        return self.cache[:, self.dc:]


def build_mla(*, name: str, contexts, heads: int, dc: int = 512, dr: int = 64, topk: int = 2048,
              kpool: int = 4, num_slots: int = 1 << 18, seed: int, holes: bool = False,
              sm_scale: float | None = None) -> MlaWorkload:
    s_val, s_slot, s_hole = (np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(3))
    ctx = np.asarray(contexts, dtype=np.int64)
    kv_len = np.where(ctx <= topk, ctx, topk + ctx % kpool).astype(np.int32)
    rows = ctx.size
    width = ((topk + kpool + 3) // 4) * 4
    slots = np.full((rows, width), -1, dtype=np.int32)
    for r in range(rows):
        n = int(kv_len[r])
        slots[r, :n] = np.sort(s_slot.choice(num_slots, size=n, replace=False))
        if holes and n > 0:
            hit = s_hole.random(n) < 0.01
            slots[r, :n][hit] = -1
            far = s_hole.random(n) < 0.002
            slots[r, :n][far] = num_slots + s_hole.integers(0, 1000, size=int(far.sum()))
    q_nope = _bf16_bits(s_val.standard_normal((rows, heads, dc)) / np.sqrt(dc))
    q_pe = _bf16_bits(s_val.standard_normal((rows, heads, dr)) / np.sqrt(dc))
    cache = _bf16_bits(s_val.standard_normal((num_slots, dc + dr)))
    # default softmax scale: 1/sqrt(192), a DeepSeek-style head of 128 no-rope + 64 rope dims
    scale = sm_scale if sm_scale is not None else 192.0 ** -0.5
    return MlaWorkload(name=name, q_nope=q_nope, q_pe=q_pe, cache=cache, slots=slots,
                       kv_len=kv_len, sm_scale=float(scale))


# Named configurations: a small mix of short and long contexts (the oracle checks it whole),
# and the decode step of the selection benchmark (8 requests x 5 rows at 128K context, whose
# rows keep topk + ctx % kpool tokens) with 16 heads of 512 + 64 dims.
MLA_CONFIGS = {
    "mla_small": dict(contexts=[1, 7, 2047, 2048, 2049, 131072], heads=16, num_slots=1 << 16, holes=True),
    "mla_decode128k": dict(contexts=[131068 + (i % 5) for i in range(40)], heads=16, num_slots=1 << 20),
}
MLA_SEEDS = {"mla_small": 3001, "mla_decode128k": 3002}


def make_mla(name: str, seed: int | None = None, **overrides) -> MlaWorkload:
    cfg = dict(MLA_CONFIGS[name], **overrides)
    return build_mla(name=name, seed=MLA_SEEDS[name] if seed is None else seed, **cfg)
