"""Where the path's state outputs land -- TEST INFRASTRUCTURE ONLY.

Plain index arithmetic, written from the definitions, that says after how many
tokens of a request each state output is taken and where it is stored.  Used
by the oracle's forward wrapper and by the tests; never by the CUDA library.

Definitions (readings of the pages where they are silent):

* Chunks are cut at ABSOLUTE positions that are multiples of chunk_size Q.  A
  request that already holds s = num_computed_tokens tokens covers absolute
  positions [s, s+L); its first chunk may be partial (it starts at s mod Q) and
  so may its last.  ("[Bugfix] Mamba2 SSD varlen bug fix initstates decay",
  Purpose and the chunk_size note: chunk_size is a power of two and does not
  change results; "Automatic prefix caching for GDN hybrid models", the
  scatter listing, which skips requests whose num_computed_tokens is not a
  multiple of chunk_size because its chunks were request-relative.  With
  absolute chunks every block boundary is a chunk end, so nothing is skipped.)
* The exported state of a chunk is the state AFTER the chunk's last token
  (the FLA-style ``h`` export named on the prefix-caching page, Kernels/layers;
  its exact semantics are pinned there by tests the page only names).
  Chunk j of request i is row first_chunk[i] + j of the export buffer;
  first_chunk is the exclusive prefix sum of the per-request chunk counts.
* Block checkpoints: for every absolute block boundary kb (a multiple of
  block_size) with s < kb <= s+L, the state after absolute token kb-1 goes to
  pool[block_table[i][kb/block_size - 1]]; a table entry < 0 means "do not
  write" (prefix-caching page, Purpose and the scatter listing).
"""
from __future__ import annotations

from dataclasses import dataclass


def request_chunk_ends(L: int, s: int, Q: int) -> list[int]:
    """Token counts (1..L) at which each chunk of a request ends.

    The request covers absolute positions [s, s+L); chunk boundaries sit at
    the multiples of Q.  An empty request has no chunks.
    """
    if Q <= 0:
        raise ValueError("chunk_size must be positive")
    ends: list[int] = []
    pos = s
    while pos < s + L:
        nxt = min((pos // Q + 1) * Q, s + L)
        ends.append(nxt - s)
        pos = nxt
    return ends


def request_block_boundaries(L: int, s: int, block_size: int) -> list[tuple[int, int]]:
    """(token count k, block-table column j) for every block boundary kb in (s, s+L].

    k = kb - s tokens of this call have been consumed at the boundary and
    j = kb / block_size - 1 is the absolute block index that ends there.
    """
    if block_size <= 0:
        return []
    out = []
    kb = (s // block_size + 1) * block_size
    while kb <= s + L:
        out.append((kb - s, kb // block_size - 1))
        kb += block_size
    return out


@dataclass
class Record:
    request: int
    k: int            # state after k tokens of this request (1..L)
    kind: str         # "chunk" or "block"
    dest: int         # export row (kind == "chunk") or pool slot (kind == "block")


def checkpoint_records(lengths, num_computed, Q, block_size=0, block_table=None,
                       export_chunks=False):
    """Every state output of one call, in request order then token order.

    Returns (records, first_chunk) where first_chunk[i] is request i's first
    row in the chunk-export buffer and first_chunk[R] the row count.
    Block-table entries < 0 produce no record.
    """
    R = len(lengths)
    first_chunk = [0] * (R + 1)
    recs: list[Record] = []
    for i in range(R):
        L = int(lengths[i])
        s = int(num_computed[i]) if num_computed is not None else 0
        ends = request_chunk_ends(L, s, Q)
        first_chunk[i + 1] = first_chunk[i] + len(ends)
        if export_chunks:
            for j, k in enumerate(ends):
                recs.append(Record(i, k, "chunk", first_chunk[i] + j))
        if block_table is not None and block_size > 0:
            for k, j in request_block_boundaries(L, s, block_size):
                if j >= len(block_table[i]):
                    raise IndexError(f"request {i} needs block-table column {j}")
                slot = int(block_table[i][j])
                if slot >= 0:
                    recs.append(Record(i, k, "block", slot))
    recs.sort(key=lambda r: (r.request, r.k))
    return recs, first_chunk
