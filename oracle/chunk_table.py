"""CPU builder of the static chunk-index table (TEST INFRASTRUCTURE).

Follows the static-grid design of the FLA RFC "Graph capture support for
prefill and training" (section "Core design"): given cu_seqlens padded to
N_max + 1 entries, every slot s < NT_max of a fixed [NT_max, 2] table holds
(sequence id, chunk ordinal inside that sequence) for a real chunk, ordered by
sequence and then by ordinal, and a sentinel otherwise. The bound
NT_max = cdiv(T_max, C) + N_max - 1 is the one the same section states.

Readings: the second column is the chunk ordinal (token start =
cu_seqlens[n] + C * ordinal); the sentinel is (-1, -1). chunk_offsets[n] is
the slot of sequence n's first chunk, with chunk_offsets[N] = total chunks.
Written as plain loops so that it can be checked by eye.
"""
from __future__ import annotations

SENTINEL = -1


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def nt_max_bound(T_max: int, N_max: int, chunk_size: int = 64) -> int:
    """Closed-form upper bound on the number of chunks (RFC "Core design")."""
    return cdiv(T_max, chunk_size) + N_max - 1


def build_chunk_table(cu_seqlens, nt_max: int, chunk_size: int = 64):
    """Return (chunk_indices as a list of [seq, ordinal] pairs of length nt_max,
    chunk_offsets as a list of N+1 ints, total number of real chunks).

    Chunks beyond nt_max (an undersized bound) are dropped from the table but
    still counted in chunk_offsets and the total."""
    cu = [int(x) for x in cu_seqlens]
    n_seq = len(cu) - 1
    table = [[SENTINEL, SENTINEL] for _ in range(nt_max)]
    offsets = [0] * (n_seq + 1)
    slot = 0
    for n in range(n_seq):
        offsets[n] = slot
        length = cu[n + 1] - cu[n]
        for c in range(cdiv(length, chunk_size)):
            if slot < nt_max:
                table[slot] = [n, c]
            slot += 1
    offsets[n_seq] = slot
    return table, offsets, slot
