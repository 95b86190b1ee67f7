"""Prefill plan oracle (test infrastructure only).

Follows generic_flare_mla_prefill_ragged_paged_plan: from the Q row offsets
(Args: input_row_offsets, shape batch+1) and the paged cache's per-sequence
cache lengths (Args: kv_collection) it fills

  buffer_row_offsets  start/end of each K entry in the ragged K/V buffer row,
  cache_offsets       start of each K entry in the paged cache,
  buffer_lengths      valid tokens per buffer row (int32),

so that the K context is consumed in buffer rows of buffer_token_size tokens
(Args: buffer_token_size; summary: "gather K/V entries into a contiguous
buffer").

Readings taken where the page is silent:
* cache_lens[b] is the prior (already cached) length; sequence b's K context
  holds L_b = cache_lens[b] + (input_row_offsets[b+1] - input_row_offsets[b])
  tokens.
* Global packing: buffer row r is the token window [r*T, (r+1)*T) of the
  batch-order concatenation of all K contexts.  buffer_row_offsets[r] holds
  B+1 ragged offsets into that row, cache_offsets[r, b] the first token of
  sequence b that row r holds (for a sequence absent from the row: L_b if it
  already finished, 0 if it has not started).
* Rows past the last used one get buffer_lengths = -1 (the only signed output
  marks unused rows); their offsets follow the same definition.

Two independent derivations are given; tests require them to agree bit for
bit and pin both to a hand-worked example.
"""
import numpy as np


def context_lengths(input_row_offsets, cache_lens):
    iro = np.asarray(input_row_offsets, dtype=np.int64)
    prior = np.asarray(cache_lens, dtype=np.int64)
    return prior + (iro[1:] - iro[:-1])


def num_rows(input_row_offsets, cache_lens, buffer_token_size):
    S = int(context_lengths(input_row_offsets, cache_lens).sum())
    T = int(buffer_token_size)
    return (S + T - 1) // T


def plan_formula(input_row_offsets, cache_lens, buffer_token_size, max_rows):
    """Closed-form windows.  Returns (bro uint32 [R_max,B+1], co uint32 [R_max,B],
    blen int32 [R_max], R)."""
    T = int(buffer_token_size)
    assert T > 0
    L = context_lengths(input_row_offsets, cache_lens)
    B = L.shape[0]
    G = np.zeros(B + 1, dtype=np.int64)          # start of each context in the packing
    for b in range(B):
        G[b + 1] = G[b] + L[b]
    S = int(G[B])
    R = (S + T - 1) // T
    bro = np.zeros((max_rows, B + 1), dtype=np.int64)
    co = np.zeros((max_rows, B), dtype=np.int64)
    blen = np.zeros(max_rows, dtype=np.int64)
    for r in range(max_rows):
        start = r * T
        for b in range(B + 1):
            bro[r, b] = min(max(G[b] - start, 0), T)
        for b in range(B):
            co[r, b] = min(max(start - G[b], 0), L[b])
        blen[r] = min(T, S - start) if r < R else -1
    return bro.astype(np.uint32), co.astype(np.uint32), blen.astype(np.int32), R


def plan_token_walk(input_row_offsets, cache_lens, buffer_token_size, max_rows):
    """Brute force: place every K token, one at a time, into buffer rows of T
    slots in batch order, counting per (row, sequence); the outputs are then
    prefix counts.  Shares nothing with plan_formula but the reading."""
    T = int(buffer_token_size)
    L = context_lengths(input_row_offsets, cache_lens)
    B = L.shape[0]
    rows_used = 0
    count = {}                                   # (row, seq) -> tokens of seq in row
    row, slot = 0, 0
    for b in range(B):
        for _ in range(int(L[b])):
            count[(row, b)] = count.get((row, b), 0) + 1
            rows_used = row + 1
            slot += 1
            if slot == T:
                row, slot = row + 1, 0
    bro = np.zeros((max_rows, B + 1), dtype=np.int64)
    co = np.zeros((max_rows, B), dtype=np.int64)
    blen = np.zeros(max_rows, dtype=np.int64)
    for r in range(max_rows):
        acc = 0
        for b in range(B):
            bro[r, b] = acc
            acc += count.get((r, b), 0)
        bro[r, B] = acc
        for b in range(B):
            co[r, b] = sum(count.get((rr, b), 0) for rr in range(r))
        blen[r] = acc if r < rows_used else -1
    return bro.astype(np.uint32), co.astype(np.uint32), blen.astype(np.int32), rows_used
