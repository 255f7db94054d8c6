"""Pins of oracle/kv_compact.py: a paged example worked by hand, the case
where a destination is an earlier step's source, the chain identity, bad
pages."""

import numpy as np

from oracle import kv_compact as C


def _cache(pages, P, W):
    # row value = 1000 * page + 10 * slot + element, so every row is recognisable
    kv = np.zeros((pages, P, W))
    for pg in range(pages):
        for sl in range(P):
            kv[pg, sl] = 1000 * pg + 10 * sl + np.arange(W)
    return kv


def test_hand_worked_paged_move():
    P, W = 2, 3
    kv = _cache(6, P, W)
    table = np.array([[4, 1, 5, 0]])          # logical pages of request 0
    # base 1: node n lives at position 1 + n; path 0 -> 2 -> 5, n = 2
    out, L, st = C.compact(kv, table, P, [1], np.array([[0, 2, 5, -1]]), [2], max_nodes=6)
    # position 1 (node 0) stays: page table[0] = 4, slot 1
    assert np.array_equal(out[4, 1], kv[4, 1])
    # position 2 <- node 2 at position 3 (page table[1] = 1, slot 1); position 2 is page 1 slot 0
    assert np.array_equal(out[1, 0], kv[1, 1])
    # position 3 <- node 5 at position 6 (page table[3] = 0, slot 0); position 3 is page 1 slot 1
    assert np.array_equal(out[1, 1], kv[0, 0])
    assert L.tolist() == [4] and st.tolist() == [0]
    changed = {(pg, sl) for pg in range(6) for sl in range(P) if not np.array_equal(out[pg, sl], kv[pg, sl])}
    assert changed == {(1, 0), (1, 1)}


def test_destination_that_is_an_earlier_source():
    # path 0 -> 1? no: 0 -> 2 -> 3: step 1 reads position 2 and step 2 writes it
    P, W = 4, 2
    kv = _cache(2, P, W)
    table = np.array([[0, 1]])
    out, L, _ = C.compact(kv, table, P, [0], np.array([[0, 2, 3]]), [2], max_nodes=4)
    assert np.array_equal(out[0, 1], kv[0, 2])      # position 1 <- node 2
    assert np.array_equal(out[0, 2], kv[0, 3])      # position 2 <- node 3 (read before overwritten)
    assert L.tolist() == [3]


def test_chain_path_is_an_identity_and_bad_pages_are_flagged():
    P, W = 4, 5
    kv = _cache(3, P, W)
    table = np.array([[2, 0, 1], [1, -1, 2]])
    out, L, st = C.compact(kv, table, P, [3, 2], np.array([[0, 1, 2, 3], [0, 1, 5, 9]]), [3, 3], max_nodes=10)
    assert np.array_equal(out, kv)        # request 0 is a chain (nothing moves), request 1 is rejected
    assert L.tolist() == [7, 2] and st.tolist() == [0, C.STATUS_BAD_PAGE]       # request 1 touches page -1
