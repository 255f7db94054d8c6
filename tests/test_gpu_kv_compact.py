"""GPU parity of accepted-path KV compaction against oracle/kv_compact.py
(a byte copy, so results are compared exactly), with paths taken from real
tree verifications, hand-made overlapping paths, chains and bad pages."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import workloads as W
from oracle import kv_compact as C
from parity_utils import host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def _cache(B, P, row_shape, need_pos, dtype, seed):
    """A paged cache with a random page table: pages shuffled across requests."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    per_req = (need_pos + P - 1) // P
    pages = B * per_req + 3
    kv = torch.randn((pages, P) + row_shape, generator=g).to(dtype)
    perm = torch.randperm(pages, generator=g)[:B * per_req].view(B, per_req).to(torch.int32)
    return kv, perm


def _run(kv, table, base, nodes, n, max_nodes):
    ref, L, st = C.compact(kv.float().numpy() if kv.dtype == torch.bfloat16 else kv.numpy(), table.numpy(), kv.shape[1],
                           base, nodes, n, max_nodes)
    d = kv.to(DEV)
    got = sv.spec_kv_compact(d, table.to(DEV), torch.tensor(base, dtype=torch.int32, device=DEV),
                             torch.tensor(nodes, dtype=torch.int32, device=DEV),
                             torch.tensor(n, dtype=torch.int32, device=DEV), max_nodes)
    out = d.cpu()
    out = out.float().numpy() if out.dtype == torch.bfloat16 else out.numpy()
    assert np.array_equal(out, ref)
    assert host(got["out_len"]).tolist() == L.tolist()
    assert host(got["status"]).tolist() == st.tolist()
    return got


@pytest.mark.parametrize("row_shape,dtype", [((64,), torch.float32), ((2, 8, 128), torch.bfloat16)])
def test_paths_from_tree_verification(row_shape, dtype):
    B, N, P = 24, 64, 16
    ti = W.eagle_tree(B=B, V=5000, seed=7800, device=DEV)
    ver = sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth)
    nodes, n = host(ver["nodes"]).astype(np.int64), host(ver["num_accepted"]).astype(np.int64)
    rng = np.random.default_rng(1)
    base = rng.integers(0, 40, size=B)
    kv, table = _cache(B, P, row_shape, int(base.max()) + N, dtype, 7801)
    assert (n > 0).any()
    _run(kv, table, base.tolist(), nodes, n.tolist(), N)


def test_overlapping_chain_and_bad_paths():
    P = 4
    kv, table = _cache(4, P, (32,), 16, torch.float32, 7802)
    nodes = np.array([[0, 2, 3, -1], [0, 1, 2, 3], [0, 3, 9, 12], [0, 5, 7, -1]])
    n = [2, 3, 3, 2]
    table[3, 1] = -1                          # request 3's node 5 sits on a missing page
    got = _run(kv, table, [0, 1, 2, 0], nodes, n, 13)
    assert host(got["status"]).tolist() == [0, 0, 0, C.STATUS_BAD_PAGE]


def test_large_rows_span_many_chunks():
    # Llama-3.1-8B-sized rows: 32 layers x (K, V) x 8 heads x 128 dims of bf16 = 128 KB per token
    B, N, P = 6, 20, 16
    kv, table = _cache(B, P, (32, 2, 8, 128), 60, torch.bfloat16, 7803)
    rng = np.random.default_rng(2)
    nodes = np.full((B, 6), -1)
    n = []
    for b in range(B):
        k = int(rng.integers(0, 6))
        path = [0] + sorted(rng.choice(np.arange(1, N), size=k, replace=False).tolist())
        nodes[b, :k + 1] = path
        n.append(k)
    _run(kv, table, rng.integers(0, 30, size=B).tolist(), nodes, n, N)
