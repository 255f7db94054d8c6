"""CPU oracle for accepted-path KV compaction, the step after tree
verification.

TEST INFRASTRUCTURE: only tests/ (and bench.py's oracle legs) use this
module; it shares no code with the CUDA library.

Sources: nanospec README, introduction (a paged KV cache, EAGLE-3 tree
speculation on Llama-3.1-8B); mini-sglang PR #134, Modifications (draft.py):
after verification the cache keeps the accepted prefix and drops the rest
("rollback() a plain cache truncation"). Reading taken for trees (the pages
describe the cache, not the kernel):
  * the verify pass wrote node n's key/value row at logical position
    seq_base[b] + n of request b (node 0 = the root, the last token already
    emitted); a logical position p lives in page page_table[b, p // P] at
    slot p % P of a cache laid out [pages, P, W] (W elements per token row,
    consecutive rows token_stride elements apart);
  * the accepted path path_nodes[b, 0..n] (node ids from tree verification,
    path_nodes[b, 0] = 0, strictly increasing since parents precede children)
    is moved so that node path_nodes[b, j] lands at position seq_base[b] + j;
  * every source row is read before any destination is written (equivalently
    j increasing: a destination is never a later source, since
    path_nodes[j'] >= j' > j), rows not on the path are left as they are,
    and the committed length becomes seq_base[b] + n + 1 (the root and the n
    accepted nodes; the bonus token has no row yet);
  * a path node outside [0, max_nodes) or a page id < 0 leaves the request
    untouched and sets status bit BAD_PAGE (256).

Parity status: pinned by tests/test_oracle_kv_compact.py (a hand-worked
paged example, the overlap case, the chain identity).
"""

from __future__ import annotations

import numpy as np

STATUS_BAD_PAGE = 256


def _slot(page_table, b, p, P):
    page = int(page_table[b, p // P])
    return page, p % P


def compact(kv, page_table, page_size, seq_base, path_nodes, num_accepted, max_nodes):
    """kv: [pages, page_size, W] array (copied). Returns (kv', new_len [B], status [B])."""
    out = np.array(kv, copy=True)
    B = len(seq_base)
    new_len = np.zeros(B, dtype=np.int64)
    status = np.zeros(B, dtype=np.int64)
    for b in range(B):
        n = int(num_accepted[b])
        nodes = [int(path_nodes[b, j]) for j in range(n + 1)]
        base = int(seq_base[b])
        ok = all(0 <= v < max_nodes for v in nodes)
        pages_needed = [(base + v) // page_size for v in nodes] + [(base + j) // page_size for j in range(n + 1)]
        ok = ok and all(0 <= q < page_table.shape[1] and int(page_table[b, q]) >= 0 for q in pages_needed)
        if not ok:
            status[b] = STATUS_BAD_PAGE
            new_len[b] = base
            continue
        rows = []
        for j in range(n + 1):                       # read every source first
            pg, sl = _slot(page_table, b, base + nodes[j], page_size)
            rows.append(out[pg, sl].copy())
        for j in range(n + 1):                       # then write the destinations
            pg, sl = _slot(page_table, b, base + j, page_size)
            out[pg, sl] = rows[j]
        new_len[b] = base + n + 1
    return out, new_len, status
