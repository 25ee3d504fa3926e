"""Partitioning one KDA forward across ranks (one process per GPU).

Every (sequence, value head) pair is an independent problem: its state never
meets another's.  A multi-GPU run therefore splits the work with no exchange
on the data path: each rank takes whole sequences (batch rows) when there are
at least as many as ranks, otherwise a contiguous block of value heads (kept
aligned to key-head groups so that each rank's q and k are a plain slice).
The host gathers outputs and final states, if it needs them, after the fact.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Shard:
    rank: int
    world: int
    batch: tuple[int, int]    # [b0, b1) rows of the batch
    heads: tuple[int, int]    # [h0, h1) value heads
    key_heads: tuple[int, int]  # [hk0, hk1) key heads used by those value heads

    @property
    def empty(self) -> bool:
        return self.batch[0] >= self.batch[1] or self.heads[0] >= self.heads[1]


def _block(n: int, world: int, rank: int) -> tuple[int, int]:
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard(B: int, H: int, HV: int, rank: int, world: int) -> Shard:
    """Rank `rank`'s part of a [B, T, H/HV, ...] forward among `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    if HV % H:
        raise ValueError("HV must be a multiple of H")
    G = HV // H
    if B >= world or H == 1 and G == 1:
        b0, b1 = _block(B, world, rank)
        return Shard(rank, world, (b0, b1), (0, HV), (0, H))
    # split key-head groups so each rank's q, k are contiguous key heads
    k0, k1 = _block(H, world, rank)
    return Shard(rank, world, (0, B), (k0 * G, k1 * G), (k0, k1))


def take(sh: Shard, q, k, v, g, beta, initial_state=None):
    """Slice the inputs (tensors or arrays laid out as in the forward) for one shard."""
    b0, b1 = sh.batch
    h0, h1 = sh.heads
    k0, k1 = sh.key_heads
    cont = lambda x: x.contiguous() if hasattr(x, "contiguous") else x.copy()
    out = (cont(q[b0:b1, :, k0:k1]), cont(k[b0:b1, :, k0:k1]), cont(v[b0:b1, :, h0:h1]),
           cont(g[b0:b1, :, h0:h1]), cont(beta[b0:b1, :, h0:h1]))
    s0 = None if initial_state is None else cont(initial_state[b0:b1, h0:h1])
    return out + (s0,)
