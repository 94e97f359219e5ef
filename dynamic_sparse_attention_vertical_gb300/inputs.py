"""Seeded synthetic inputs for the sparse prefill attention path.

This module only draws random tensors and plants structure into them. It holds
none of the method's arithmetic (no logits, no softmax, no top-k), so that both
the CUDA path and the CPU oracle can be fed the same inputs without sharing any
computation.

Shapes follow the long-context decoder layer the MInference pages use as their
workload (LLaMA-3-8B-1M: 32 query heads, 8 KV heads, head dim 128, 4K..1M
tokens); tensors are ``[heads, seqlen, d]`` bf16.

Three families of inputs:

``literal``
    Q, K, V ~ N(0, 1/d), plus per KV head a few planted key columns and planted
    diagonal offsets.  A planted column c draws u ~ N(0, I/d), adds 4u to
    K[c] and u to every query row of every q-head in the group.  A planted
    offset o draws, for every row i >= o, a fresh r_i ~ N(0, I/d), adds r_i
    to Q[i] of every q-head in the group and 4 r_i to K[i - o].  All
    additions are done in fp32 before one round-to-nearest-even to bf16.

``margin`` (margin-planted)
    The last ``last_q`` query rows of every q-head are scaled one-hot vectors
    beta * e_i in the first ``last_q`` dimensions.  A planted key column gets
    alpha_v in all of those dimensions; a planted offset o gets alpha_s in
    dimension i of key N - last_q + i - o.  Every other key is zero in those
    dimensions, so the estimation scores of the planted columns and offsets are
    separated from all others by a wide, known margin and the expected index
    sets are the planted sets themselves.

``local``
    The literal inputs plus a low-frequency rotary pair in two reserved
    dimensions, so that attention to nearby keys is slightly favoured and the
    highest-scoring diagonals cluster at small offsets, the locality that real
    heads show.

``grid`` (grid-planted)
    As ``margin``, but the planted key columns are a whole lattice j = phi
    (mod sigma): the last ``last_q`` query rows attend to it, so its columns
    carry almost all of the vertical score.

``modality`` (modality-planted, two modalities)
    Tokens are split into runs of modality 0 and 1.  For each modality m the
    ``last_q`` rows that end at its last token are one-hot in the dimensions
    64 m .. 64 m + 63, and the keys of its planted columns and offsets carry
    the planted values in those dimensions only, so each modality's window
    selects its own planted sets with a wide margin.

``pattern heads`` (for the offline pattern search)
    Three heads, one KV head each, each shaped like one of the slides' three
    patterns: head 0 attends to a sink (the first keys) and a local window,
    head 1 to scattered planted columns and diagonals, head 2 to whole 64x64
    blocks chosen by a per-block topic.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

__all__ = [
    "Inputs",
    "kv_group",
    "literal_inputs",
    "margin_inputs",
    "local_inputs",
    "pattern_head_inputs",
    "grid_inputs",
    "modality_inputs",
    "uniform_choice",
]


@dataclasses.dataclass
class Inputs:
    """A generated layer: tensors plus what was planted.

    ``planted_cols[g]`` / ``planted_offsets[g]`` are sorted int64 tensors (CPU)
    of the structure planted into KV head ``g``; they are shared by the q-heads
    of that group.
    """

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    planted_cols: List[torch.Tensor]
    planted_offsets: List[torch.Tensor]
    seed: int
    kind: str

    @property
    def shape(self):
        return tuple(self.q.shape)


def kv_group(h: int, Hq: int, Hkv: int) -> int:
    """KV head serving q-head ``h``: consecutive grouping, ``h // (Hq // Hkv)``."""
    return h // (Hq // Hkv)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def uniform_choice(n_pick: int, lo: int, hi: int, gen: torch.Generator) -> torch.Tensor:
    """``n_pick`` distinct integers drawn uniformly from ``[lo, hi)``, sorted (CPU int64)."""
    span = hi - lo
    if n_pick > span:
        raise ValueError(f"cannot pick {n_pick} distinct values from a range of {span}")
    perm = torch.randperm(span, generator=gen, device=gen.device)[:n_pick]
    return (perm.to("cpu") + lo).sort().values


def _randn(shape, gen, device, scale):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * scale


def literal_inputs(
    Hq: int,
    Hkv: int,
    N: int,
    d: int = 128,
    n_cols: int = 8,
    n_offsets: int = 4,
    seed: int = 1,
    device: str = "cpu",
    strength: float = 4.0,
) -> Inputs:
    """N(0, 1/d) Q/K/V with planted key columns and diagonal offsets per KV head.

    Columns are drawn from [64, N-64), offsets from [64, N-64].  Generated
    one KV group at a time in fp32 and rounded once to bf16.
    """
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g_per = Hq // Hkv
    gen = _gen(device, seed)
    sd = 1.0 / math.sqrt(d)
    q = torch.empty((Hq, N, d), dtype=torch.bfloat16, device=device)
    k = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    cols_all, offs_all = [], []
    lo, hi_c, hi_o = 64, max(64, N - 64), max(65, N - 64 + 1)
    for grp in range(Hkv):
        kf = _randn((N, d), gen, device, sd)
        v[grp] = _randn((N, d), gen, device, sd).to(torch.bfloat16)
        qf = _randn((g_per, N, d), gen, device, sd)
        cols = uniform_choice(min(n_cols, max(0, hi_c - lo)), lo, hi_c, gen) if n_cols else torch.empty(0, dtype=torch.int64)
        offs = uniform_choice(min(n_offsets, max(0, hi_o - lo)), lo, hi_o, gen) if n_offsets else torch.empty(0, dtype=torch.int64)
        for c in cols.tolist():
            u = _randn((d,), gen, device, sd)
            kf[c] += strength * u
            qf += u
        for o in offs.tolist():
            r = _randn((N - o, d), gen, device, sd)
            qf[:, o:, :] += r
            kf[: N - o] += strength * r
            del r
        k[grp] = kf.to(torch.bfloat16)
        q[grp * g_per:(grp + 1) * g_per] = qf.to(torch.bfloat16)
        del kf, qf
        cols_all.append(cols)
        offs_all.append(offs)
    return Inputs(q, k, v, cols_all, offs_all, seed, "literal")


def margin_inputs(
    Hq: int,
    Hkv: int,
    N: int,
    k_v: int,
    k_s: int,
    d: int = 128,
    last_q: int = 64,
    seed: int = 101,
    device: str = "cpu",
    beta: float = 8.0,
    alpha_v: float = 9.5,
    alpha_s: float = 8.5,
) -> Inputs:
    """Inputs whose top-k_v columns and top-k_s offsets are the planted sets.

    Per KV head, ``k_v`` columns are planted in [64, N-64) and ``k_s`` offsets
    in [0, N-last_q] (every planted offset is seen by all ``last_q`` rows).
    Dimensions ``last_q..d`` of keys carry N(0, 1/d) noise, dimensions
    ``0..last_q`` only the planted structure; the last ``last_q`` query rows
    are ``beta * e_i``.  All other query rows are N(0, 1/d).  V ~ N(0, 1/d).
    Values beta=8, alpha=8.5/9.5 are exact in bf16.
    """
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if d < 2 * last_q:
        raise ValueError("margin inputs need d >= 2*last_q")
    g_per = Hq // Hkv
    gen = _gen(device, seed)
    sd = 1.0 / math.sqrt(d)
    q = torch.empty((Hq, N, d), dtype=torch.bfloat16, device=device)
    k = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    cols_all, offs_all = [], []
    rows = torch.arange(last_q, device=device)
    for grp in range(Hkv):
        kf = _randn((N, d), gen, device, sd)
        kf[:, :last_q] = 0.0
        cols = uniform_choice(k_v, 64, N - 64, gen)
        offs = uniform_choice(k_s, 0, N - last_q + 1, gen)
        kf[cols.to(device), :last_q] += alpha_v
        for o in offs.tolist():
            keys = N - last_q + rows - o           # key hit by row i on diagonal o
            kf[keys, rows] += alpha_s
        k[grp] = kf.to(torch.bfloat16)
        v[grp] = _randn((N, d), gen, device, sd).to(torch.bfloat16)
        qf = _randn((g_per, N, d), gen, device, sd)
        qf[:, N - last_q:, :] = 0.0
        qf[:, N - last_q + rows, rows] = beta
        q[grp * g_per:(grp + 1) * g_per] = qf.to(torch.bfloat16)
        cols_all.append(cols)
        offs_all.append(offs)
    return Inputs(q, k, v, cols_all, offs_all, seed, "margin")


def local_inputs(
    Hq: int,
    Hkv: int,
    N: int,
    d: int = 128,
    n_cols: int = 16,
    n_offsets: int = 8,
    seed: int = 1,
    device: str = "cpu",
    period: int = 16384,
    amplitude: float = 1.0,
) -> Inputs:
    """``literal_inputs`` plus a low-frequency rotary pair in dims (d-2, d-1).

    Query row i gets a*(cos(i w), sin(i w)) and key row j gets
    a*(cos(j w), sin(j w)) with w = pi / (2 * period); the product of the two
    pairs is a^2 cos((i-j) w), largest at small offsets and falling to zero at
    ``period`` tokens.  ``amplitude`` is the size of that logit term in nats
    once the 1/sqrt(d) softmax scale is applied.
    """
    base = literal_inputs(Hq, Hkv, N, d, n_cols, n_offsets, seed, device)
    w = math.pi / (2.0 * period)
    a = math.sqrt(amplitude * math.sqrt(d))
    pos = torch.arange(N, device=device, dtype=torch.float64) * w
    rot = torch.stack([torch.cos(pos), torch.sin(pos)], dim=-1).to(torch.float32) * a
    q = base.q.clone()
    k = base.k.clone()
    q[:, :, d - 2:] = rot.to(torch.bfloat16)
    k[:, :, d - 2:] = rot.to(torch.bfloat16)
    return Inputs(q, k, base.v, base.planted_cols, base.planted_offsets, seed, "local")


def _logit_scale(nats: float, d: int) -> float:
    """Size a of two unit-direction entries whose product a*a is ``nats`` after the 1/sqrt(d) scale."""
    return math.sqrt(nats * math.sqrt(d))


def pattern_head_inputs(
    N: int,
    d: int = 128,
    seed: int = 1,
    device: str = "cpu",
    sink: int = 128,
    window: int = 1024,
    n_cols: int = 24,
    offsets=(700, 1900),
    n_topics: int = 12,
    nats: float = 10.0,
) -> Inputs:
    """Three single-KV-head heads shaped like the three patterns (see the module doc).

    Every head starts from Q, K, V ~ N(0, 1/d).  Head 0: keys j < ``sink`` carry a
    sink direction every query shares (+``nats``), and 16 rotary pairs with
    frequencies spread over (0, pi / ``window``] add sum_f cos(f (i - j)) * nats/16:
    ``nats`` at distance 0, positive up to about ``window`` tokens, small and not
    recurring beyond.  Head 1: ``n_cols`` key columns drawn from [64, N) each get their
    own basis direction (dims 0 ..), which every query carries (+``nats``), and
    for each offset o in ``offsets`` every row i >= o and key i - o share a fresh
    random unit direction in the upper half of the dims (+``nats``).  Head 2:
    every 64-row block of queries and every 64-key block gets one of
    ``n_topics`` random unit directions, and a query block attends (+``nats``)
    to the key blocks of its own topic.  The planted columns and offsets of
    head 1 are recorded in slot 1; the other slots record none.
    """
    if n_cols > d // 2:
        raise ValueError("n_cols must fit in the lower half of the head dimension")
    gen = _gen(device, seed)
    sd = 1.0 / math.sqrt(d)
    q = torch.empty((3, N, d), dtype=torch.bfloat16, device=device)
    k = torch.empty((3, N, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((3, N, d), dtype=torch.bfloat16, device=device)
    a = _logit_scale(nats, d)
    # head 0: sink + local window
    qf = _randn((N, d), gen, device, sd)
    kf = _randn((N, d), gen, device, sd)
    qf[:, d - 34] = a
    kf[:sink, d - 34] += a
    pos = torch.arange(N, device=device, dtype=torch.float64)
    for f in range(16):
        ang = pos * (math.pi / window) * (f + 1) / 16.0
        rot = torch.stack([torch.cos(ang), torch.sin(ang)], dim=-1).to(torch.float32) * (a / 4.0)
        qf[:, d - 32 + 2 * f: d - 30 + 2 * f] = rot
        kf[:, d - 32 + 2 * f: d - 30 + 2 * f] = rot
    q[0], k[0] = qf.to(torch.bfloat16), kf.to(torch.bfloat16)
    v[0] = _randn((N, d), gen, device, sd).to(torch.bfloat16)
    # head 1: vertical columns + long-range diagonals
    qf = _randn((N, d), gen, device, sd)
    kf = _randn((N, d), gen, device, sd)
    cols = uniform_choice(n_cols, 64, N, gen)
    for i, c in enumerate(cols.tolist()):
        qf[:, i] += a
        kf[c, i] += a
    half = d // 2
    offs = torch.tensor(sorted(o for o in offsets if o < N), dtype=torch.int64)
    for o in offs.tolist():
        f = _randn((N - o, half), gen, device, 1.0)
        f = f / f.norm(dim=1, keepdim=True) * a
        qf[o:, half:] += f
        kf[: N - o, half:] += f
    q[1], k[1] = qf.to(torch.bfloat16), kf.to(torch.bfloat16)
    v[1] = _randn((N, d), gen, device, sd).to(torch.bfloat16)
    # head 2: block topics
    nb = (N + 63) // 64
    dirs = _randn((n_topics, d), gen, device, 1.0)
    dirs = dirs / dirs.norm(dim=1, keepdim=True)
    tq = torch.randint(0, n_topics, (nb,), generator=gen, device=device)
    tk = torch.randint(0, n_topics, (nb,), generator=gen, device=device)
    rows = torch.arange(N, device=device) // 64
    qf = _randn((N, d), gen, device, sd) + a * dirs[tq[rows]]
    kf = _randn((N, d), gen, device, sd) + a * dirs[tk[rows]]
    q[2], k[2] = qf.to(torch.bfloat16), kf.to(torch.bfloat16)
    v[2] = _randn((N, d), gen, device, sd).to(torch.bfloat16)
    empty = torch.empty(0, dtype=torch.int64)
    return Inputs(q, k, v, [empty, cols, empty], [empty, offs, empty], seed, "pattern_heads")


def grid_inputs(
    Hq: int,
    Hkv: int,
    N: int,
    sigma: int,
    phi: int,
    d: int = 128,
    last_q: int = 64,
    seed: int = 301,
    device: str = "cpu",
    beta: float = 8.0,
    alpha: float = 12.0,
) -> Inputs:
    """Inputs whose last ``last_q`` query rows attend to the lattice j = phi (mod sigma).

    Dimensions ``0..last_q`` of every lattice key are ``alpha`` and of every other key
    zero; the last ``last_q`` query rows are ``beta * e_i``; all other values are
    N(0, 1/d).  ``planted_cols[g]`` holds the lattice, ``planted_offsets[g]`` is empty.
    """
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g_per = Hq // Hkv
    gen = _gen(device, seed)
    sd = 1.0 / math.sqrt(d)
    q = torch.empty((Hq, N, d), dtype=torch.bfloat16, device=device)
    k = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    lattice = torch.arange(phi, N, sigma, dtype=torch.int64)
    rows = torch.arange(last_q, device=device)
    for grp in range(Hkv):
        kf = _randn((N, d), gen, device, sd)
        kf[:, :last_q] = 0.0
        kf[lattice.to(device), :last_q] = alpha
        k[grp] = kf.to(torch.bfloat16)
        v[grp] = _randn((N, d), gen, device, sd).to(torch.bfloat16)
        qf = _randn((g_per, N, d), gen, device, sd)
        qf[:, N - last_q:, :] = 0.0
        qf[:, N - last_q + rows, rows] = beta
        q[grp * g_per:(grp + 1) * g_per] = qf.to(torch.bfloat16)
    return Inputs(q, k, v, [lattice] * Hkv, [torch.empty(0, dtype=torch.int64)] * Hkv, seed, "grid")


def modality_inputs(
    Hq: int,
    Hkv: int,
    runs,
    k_v: int,
    k_s: int,
    last_q: int = 64,
    seed: int = 311,
    device: str = "cpu",
    beta: float = 8.0,
    alpha_v: float = 9.5,
    alpha_s: float = 8.5,
):
    """Two-modality inputs with planted index sets per modality (d = 128).

    ``runs``: [(modality, length), ...] in token order, modalities 0 and 1.  Each
    modality's last run must hold at least ``last_q`` tokens and the two windows of
    ``last_q`` rows ending at the modalities' last tokens must not overlap.  Returns
    (inputs, modality ids int32 [N] on ``device``, {m: (cols, offsets)} planted per
    modality; the same sets for every KV head).
    """
    d = 128
    mod = torch.cat([torch.full((n,), m, dtype=torch.int32) for m, n in runs])
    N = int(mod.numel())
    ends = {m: int(torch.nonzero(mod == m)[-1]) + 1 for m in (0, 1)}
    for m in (0, 1):
        if not bool((mod[ends[m] - last_q:ends[m]] == m).all()):
            raise ValueError("each modality's last run needs at least last_q tokens")
    if abs(ends[0] - ends[1]) < last_q:
        raise ValueError("the two estimation windows overlap")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g_per = Hq // Hkv
    gen = _gen(device, seed)
    sd = 1.0 / math.sqrt(d)
    planted = {}
    for m in (0, 1):
        R = ends[m]
        planted[m] = (uniform_choice(k_v, 64, R - 64, gen), uniform_choice(k_s, 0, R - last_q + 1, gen))
    q = torch.empty((Hq, N, d), dtype=torch.bfloat16, device=device)
    k = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=device)
    rows = torch.arange(last_q, device=device)
    for grp in range(Hkv):
        kf = torch.zeros((N, d), dtype=torch.float32, device=device)
        qf = _randn((g_per, N, d), gen, device, sd)
        for m in (0, 1):
            R, dims = ends[m], 64 * m + rows
            cols, offs = planted[m]
            kf[cols.to(device)[:, None], dims[None, :]] += alpha_v
            for o in offs.tolist():
                kf[R - last_q + rows - o, dims] += alpha_s
            qf[:, R - last_q:R, :] = 0.0
            qf[:, R - last_q + rows, dims] = beta
        k[grp] = kf.to(torch.bfloat16)
        v[grp] = _randn((N, d), gen, device, sd).to(torch.bfloat16)
        q[grp * g_per:(grp + 1) * g_per] = qf.to(torch.bfloat16)
    x = Inputs(q, k, v, [planted[0][0]] * Hkv, [planted[0][1]] * Hkv, seed, "modality")
    return x, mod.to(device), planted
