"""Split one gdn_chunk_fwd call over P ranks (one GPU each) and put the
results back together.

The (sequence, value head) chains of the chunked forward pass are
independent: no chain reads another's tokens or state.  So one call splits
with no exchange between ranks, in either of two ways:

* by qk-head groups -- rank r takes a contiguous range of the Hqk qk heads and
  the G = Hv / Hqk value heads that read each of them (value head h reads qk
  head h // G), with the matching slices of g, beta, h0 and the outputs;
* by whole sequences -- rank r takes a contiguous range of sequences, cut at
  cu_seqlens boundaries (or batch rows) so that the ranks' token counts are as
  equal as whole sequences allow, with its slice of h0 / ht and its own,
  rebased cu_seqlens.

Only index bookkeeping lives here (which rows and heads a rank owns, slicing,
reassembly); every step of the operator runs in the library's kernels (or, in
the CPU tests, in the oracle).  A sequence-parallel split of one long sequence
would need an exchange of the segments' affine state maps; within one GPU the
chunk-parallel path does that, and across ranks it is not built.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import torch


@dataclass(frozen=True)
class HeadPart:
    """Rank's qk heads [hq0, hq1) and value heads [hv0, hv1)."""
    hq0: int
    hq1: int
    hv0: int
    hv1: int


@dataclass(frozen=True)
class SeqPart:
    """Rank's sequences [n0, n1) and packed token rows [t0, t1) (for a
    fixed-length batch: batch rows [n0, n1) and all tokens)."""
    n0: int
    n1: int
    t0: int
    t1: int


def _even_cuts(total: int, parts: int) -> list[int]:
    return [(total * r) // parts for r in range(parts + 1)]


def head_part(Hqk: int, Hv: int, world: int, rank: int) -> HeadPart:
    """Contiguous qk-head range of `rank` (as equal as whole qk heads allow)
    and the value heads that read those qk heads."""
    if Hv % Hqk:
        raise ValueError("Hv must be a multiple of Hqk")
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    G = Hv // Hqk
    cuts = _even_cuts(Hqk, world)
    hq0, hq1 = cuts[rank], cuts[rank + 1]
    return HeadPart(hq0, hq1, hq0 * G, hq1 * G)


def seq_part(world: int, rank: int, B: int, T: int, cu_seqlens: Optional[Sequence[int]] = None) -> SeqPart:
    """Contiguous range of whole sequences of `rank`.  Packed batches
    (cu_seqlens given, host list of N + 1 offsets) are cut where the running
    token count first reaches rank / world of the total; fixed-length batches
    by batch rows."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    if cu_seqlens is None:
        cuts = _even_cuts(B, world)
        return SeqPart(cuts[rank], cuts[rank + 1], 0, T)
    cu = [int(c) for c in cu_seqlens]
    N, total = len(cu) - 1, cu[-1]
    if cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("malformed cu_seqlens")

    def first_seq_at(target: int) -> int:
        # first sequence index n with cu[n] >= target (all of N for target > total)
        for n in range(N + 1):
            if cu[n] >= target:
                return n
        return N

    bounds = [0] + [first_seq_at((total * r + world - 1) // world) for r in range(1, world)] + [N]
    for r in range(1, world + 1):
        bounds[r] = max(bounds[r], bounds[r - 1])
    n0, n1 = bounds[rank], bounds[rank + 1]
    return SeqPart(n0, n1, cu[n0], cu[n1])


def slice_heads(x: dict, part: HeadPart) -> dict:
    """The sub-problem of rank `part` from the full inputs x (keys as in
    inputs.make_inputs: q, k [B,T,Hqk,K]; v [B,T,Hv,V]; g, beta [B,T,Hv];
    h0 [N,Hv,K,V] or None; cu_seqlens, scale, C, N unchanged)."""
    out = dict(x)
    for name in ("q", "k"):
        out[name] = x[name][:, :, part.hq0:part.hq1].contiguous()
    for name in ("v", "g", "beta"):
        out[name] = x[name][:, :, part.hv0:part.hv1].contiguous()
    out["h0"] = x["h0"][:, part.hv0:part.hv1].contiguous() if x["h0"] is not None else None
    return out


def slice_sequences(x: dict, part: SeqPart) -> dict:
    """The sub-problem of rank `part` (whole sequences) with its own
    cu_seqlens rebased to start at 0."""
    out = dict(x)
    cu = x.get("cu_seqlens")
    if cu is None:
        for name in ("q", "k", "v", "g", "beta"):
            out[name] = x[name][part.n0:part.n1].contiguous()
        out["N"] = part.n1 - part.n0
    else:
        for name in ("q", "k", "v", "g", "beta"):
            out[name] = x[name][:, part.t0:part.t1].contiguous()
        out["cu_seqlens"] = (cu[part.n0:part.n1 + 1] - cu[part.n0]).contiguous()
        out["N"] = part.n1 - part.n0
    out["h0"] = x["h0"][part.n0:part.n1].contiguous() if x["h0"] is not None else None
    return out


def assemble_heads(parts: Sequence[HeadPart], outs: Sequence[tuple]) -> tuple:
    """Full (o, ht) from every rank's (o, ht) of a head split (in rank order)."""
    o = torch.cat([o_r for o_r, _ in outs], dim=2)
    hts = [ht_r for _, ht_r in outs]
    ht = torch.cat(hts, dim=1) if all(h is not None for h in hts) else None
    assert o.shape[2] == parts[-1].hv1
    return o, ht


def assemble_sequences(parts: Sequence[SeqPart], outs: Sequence[tuple], packed: bool) -> tuple:
    """Full (o, ht) from every rank's (o, ht) of a sequence split (in rank
    order; packed: o rows are concatenated along the token axis)."""
    o = torch.cat([o_r for o_r, _ in outs], dim=1 if packed else 0)
    hts = [ht_r for _, ht_r in outs]
    ht = torch.cat(hts, dim=0) if all(h is not None for h in hts) else None
    assert (ht is None) or ht.shape[0] == parts[-1].n1
    return o, ht
