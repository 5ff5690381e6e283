"""Seeded synthetic inputs shaped like the workloads of the packed-attention pages.

This module holds no attention arithmetic: it only draws document lengths,
lays out document-id maps and draws Gaussian tensors. It is the one piece of
code that both the CUDA path's tests/benchmark and the CPU oracle consume.

Recipe:
  * document lengths come from ``numpy.random.default_rng(seed)``;
  * fill rule: draw a length, append it while it still fits in the row, stop at
    the first one that does not and pad the rest of the row with id 0;
  * documents are numbered 1, 2, ... in order; padding is id 0 (the pages'
    padding id);
  * tensors are ``torch.randn`` in fp32 from ``torch.Generator().manual_seed``,
    times an optional factor, rounded to bf16 (round-to-nearest-even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAD_DOC_ID = 0


def doc_lengths(kind: str, total: int, seed: int) -> list[int]:
    """Draw document lengths by the fill rule for one row of ``total`` tokens.

    kind:
      * ``"uniform64_2048"``: integers uniform in [64, 2048];
      * ``"lognormal1024"``: lognormal with median 1024 and sigma 1.0, rounded,
        clipped to [32, 8192];
      * ``"pareto256"``: floor(256 * (1 - U) ** (-1 / 1.2)), clipped to [256, 32768];
      * ``"uniform16_64"``: integers uniform in [16, 64] (short documents).
    """
    rng = np.random.default_rng(seed)
    out: list[int] = []
    used = 0
    while True:
        if kind == "uniform64_2048":
            n = int(rng.integers(64, 2049))
        elif kind == "lognormal1024":
            n = int(round(float(rng.lognormal(mean=math.log(1024.0), sigma=1.0))))
            n = min(max(n, 32), 8192)
        elif kind == "uniform16_64":
            n = int(rng.integers(16, 65))
        elif kind == "pareto256":
            u = float(rng.random())
            n = int(math.floor(256.0 * (1.0 - u) ** (-1.0 / 1.2)))
            n = min(max(n, 256), 32768)
        else:
            raise ValueError(f"unknown length distribution {kind!r}")
        if used + n > total:
            break
        out.append(n)
        used += n
    return out


def doc_ids_from_lengths(lengths: list[int], total: int) -> np.ndarray:
    """One row of ``total`` ids: document i (1-based) for its run, 0 after the last one."""
    ids = np.zeros(total, dtype=np.int32)
    pos = 0
    for i, n in enumerate(lengths):
        ids[pos:pos + n] = i + 1
        pos += n
    return ids


def randn16(shape, seed: int, factor: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    """Seeded N(0, 1) * factor in fp32, rounded to a 16-bit type (bf16 or fp16, RNE)."""
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if factor != 1.0:
        x = x * factor
    return x.to(dtype)


def randn_bf16(shape, seed: int, factor: float = 1.0) -> torch.Tensor:
    return randn16(shape, seed, factor, torch.bfloat16)


@dataclass
class Workload:
    """One synthetic problem, CPU tensors. Layout: packed [T, H, D] unless dense."""

    name: str
    kind: str  # "dense" or "document"
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor
    scale: float
    causal: bool = True
    window: int | None = None
    doc_ids: np.ndarray | None = None  # [B, Sk]
    q_global_start: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def dims(self):
        return dict(Hq=self.q.shape[-2] if self.kind != "dense" else self.q.shape[1],
                    Dqk=self.q.shape[-1], Dv=self.v.shape[-1])


def _tensors(seed, q_shape, k_shape, v_shape, o_shape, factor=1.0):
    # four independent streams derived from one seed
    return (randn_bf16(q_shape, seed * 4 + 0, factor), randn_bf16(k_shape, seed * 4 + 1, factor),
            randn_bf16(v_shape, seed * 4 + 2, factor), randn_bf16(o_shape, seed * 4 + 3, factor))


def dense_workload(B, Hq, Hkv, Nq, Nk, Dqk, Dv, seed=0, factor=1.0, causal=True, name="dense"):
    """Dense [B, H, N, D] tensors."""
    q, k, v, do = _tensors(seed, (B, Hq, Nq, Dqk), (B, Hkv, Nk, Dqk), (B, Hkv, Nk, Dv),
                           (B, Hq, Nq, Dv), factor)
    return Workload(name, "dense", q, k, v, do, 1.0 / math.sqrt(Dqk), causal)


def document_workload(lengths_kind, Sk, Hq, Hkv, Dqk, Dv, seed=0, q_global_start=0, q_length=None,
                      window=None, name="document"):
    """One packed row of ``Sk`` tokens; queries are the shard [q0, q0 + Lq).

    Returns packed tensors q [Lq, Hq, Dqk], k [Sk, Hkv, Dqk], v [Sk, Hkv, Dv],
    dout [Lq, Hq, Dv] and doc_ids [1, Sk].
    """
    Lq = Sk - q_global_start if q_length is None else q_length
    lengths = doc_lengths(lengths_kind, Sk, seed)
    ids = doc_ids_from_lengths(lengths, Sk)[None, :]
    q, k, v, do = _tensors(seed, (Lq, Hq, Dqk), (Sk, Hkv, Dqk), (Sk, Hkv, Dv), (Lq, Hq, Dv))
    w = Workload(name, "document", q, k, v, do, 1.0 / math.sqrt(Dqk), True, window, ids,
                 q_global_start)
    w.extra["lengths"] = lengths
    return w


def config(n: int, seed: int = 0) -> Workload:
    """The five workload shapes (1-based numbering).

    1. dense causal, B=1, Hq=2, Hkv=1, N=128, D=64 (the small case);
    2. packed document-causal, 8192 tokens, lengths uniform in [64, 2048], Hq=16, Hkv=4, D=128;
    3. dense causal, B=2, Hq=8, Hkv=2, N=4096, D=512, inputs times 0.5;
    4. 16384-token row, lognormal lengths (median 1024), queries 8192..16383, Dqk=192, Dv=128,
       Hq=Hkv=16;
    5. 65536 tokens, Pareto(1.2) lengths in [256, 32768], Hq=32, Hkv=8, D=128, left window 4096,
       plus a run without window of the query shard 32768..65535 split into a local and a cross
       key chunk (``extra["cross_split"]``);
    6. short documents: 65536 tokens, lengths uniform in [16, 64], Hq=32, Hkv=8, D=128 (the
       workload that packing a KV head's query heads into one tile is for).
    """
    if n == 1:
        return dense_workload(1, 2, 1, 128, 128, 64, 64, seed, name="cfg1_dense_causal_n128_d64")
    if n == 2:
        return document_workload("uniform64_2048", 8192, 16, 4, 128, 128, seed,
                                 name="cfg2_doc_causal_t8192_d128")
    if n == 3:
        return dense_workload(2, 8, 2, 4096, 4096, 512, 512, seed, factor=0.5,
                              name="cfg3_dense_causal_n4096_d512")
    if n == 4:
        return document_workload("lognormal1024", 16384, 16, 16, 192, 128, seed, q_global_start=8192,
                                 name="cfg4_doc_causal_shard_dqk192_dv128")
    if n == 5:
        w = document_workload("pareto256", 65536, 32, 8, 128, 128, seed, window=4096,
                              name="cfg5_doc_causal_t65536_w4096")
        # the second half of the row is the query shard of the cross-chunk run:
        # keys [32768, 65536) are its local chunk, keys [0, 32768) the cross chunk
        w.extra["cross_split"] = 32768
        return w
    if n == 6:
        return document_workload("uniform16_64", 65536, 32, 8, 128, 128, seed,
                                 name="short_docs_t65536_len16_64_d128")
    raise ValueError(f"no workload {n}")


def small_document_workload(Sk, Hq, Hkv, Dqk, Dv, seed, q_global_start=0, q_length=None,
                            window=None, min_len=1, max_len=None, pad_tail=0):
    """Small random document maps for parity tests: lengths uniform in [min_len, max_len]."""
    rng = np.random.default_rng(10_000 + seed)
    max_len = max_len or Sk
    lengths = []
    used = 0
    body = Sk - pad_tail
    while True:
        n = int(rng.integers(min_len, max_len + 1))
        if used + n > body:
            break
        lengths.append(n)
        used += n
    ids = doc_ids_from_lengths(lengths, Sk)[None, :]
    Lq = Sk - q_global_start if q_length is None else q_length
    q, k, v, do = _tensors(seed, (Lq, Hq, Dqk), (Sk, Hkv, Dqk), (Sk, Hkv, Dv), (Lq, Hq, Dv))
    w = Workload("small_document", "document", q, k, v, do, 1.0 / math.sqrt(Dqk), True, window, ids,
                 q_global_start)
    w.extra["lengths"] = lengths
    return w
