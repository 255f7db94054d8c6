"""GPU parity of the stochastic tree call's two device paths against the
float64 oracle.

* The cluster path (rows on 16-byte boundaries whose chunks fit one cluster):
  the row merges, the walk and the draw run in one kernel, one cluster of
  CTAs per request, sharing the walk's result and the chunk sums through
  distributed shared memory.
* The three-kernel path (decide, chunk sums, pick), which rows off a 16-byte
  boundary and rows of more chunks than a cluster holds take.

Cases: a row end inside a 16-byte vector (the copy's extra elements masked),
a copy cut back at the buffer's end (elements read from global memory), one
chunk per row (most CTAs of the cluster hold none), the most chunks a
cluster holds (six per CTA) and one past it, rejected tokens spread over
many chunks and CTAs, a root alone, a depth cap of 0, and more nodes than the
staged merge holds.
"""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import workloads as W
from oracle import spec_oracle as O
from parity_utils import compare, f64, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
CLUSTER_MAX_CHUNKS = 8 * 6     # CTAs per request x chunks one CTA holds


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def _placed(x, off, pad):
    """x [B, N, V] copied into a flat buffer at element offset `off` with row
    pitch V + pad; returns the strided [B, N, V] view."""
    B, N, V = x.shape
    pitch = V + pad
    buf = torch.full((off + B * N * pitch,), float("nan"), dtype=x.dtype, device=x.device)
    view = buf[off: off + B * N * pitch].view(B, N, pitch)[:, :, :V]
    view.copy_(x)
    return view


def _chunks(V, dtype):
    per = 16384 // torch.tensor([], dtype=dtype).element_size()
    return (V + per - 1) // per


def _cluster_path(view):
    es = view.element_size()
    return view.data_ptr() % 16 == 0 and (view.stride(1) * es) % 16 == 0 and \
        _chunks(view.shape[2], view.dtype) <= CLUSTER_MAX_CHUNKS


RULES = [(O.RULE_EXACT, 0.0, 1.0), (O.RULE_POWER, 0.0, 0.3), (O.RULE_RELAXED, 0.1, 1.0)]


@pytest.mark.parametrize("dtype,V,off,pad,cluster", [
    (torch.bfloat16, 128256, 0, 0, True),     # 16 chunks: two per CTA
    (torch.bfloat16, 20011, 0, 5, True),      # row end inside a vector; last copy cut back
    (torch.bfloat16, 20011, 3, 2, False),     # rows off the 16-byte boundary
    (torch.float32, 9001, 0, 3, True),
    (torch.float32, 9001, 1, 3, False),
    (torch.bfloat16, 300, 0, 4, True),        # one chunk: seven CTAs hold none
    (torch.float32, 196608, 0, 0, True),      # 48 chunks: six per CTA
    (torch.float32, 196612, 0, 0, False),     # 49 chunks: past the cluster
])
def test_stochastic_tree_paths(dtype, V, off, pad, cluster):
    B = 4 if V > 100000 else 8
    ti = W.eagle_tree(B=B, V=V, dtype=dtype, seed=8100 + V + off, device=DEV)
    x = _placed(ti.target, off, pad) if (off or pad) else ti.target
    assert _cluster_path(x) == cluster
    xr = f64(ti.target)
    for rule, tau, alpha in RULES:
        got = sv.spec_verify_tree(x, ti.node_tokens, ti.parents, ti.max_depth, temperature=1.0,
                                  uniforms=ti.uniforms, rule=rule, tau=tau, alpha=alpha)
        ref = O.verify_tree(xr, host(ti.node_tokens), host(ti.parents), ti.max_depth, 1.0,
                            f64(ti.uniforms), rule=rule, tau=tau, alpha=alpha)
        compare(got, ref, stochastic=True)


@pytest.mark.parametrize("V,children", [(128256, 70), (128256, 200), (300, 70)])
def test_rejected_tokens_across_chunks(V, children):
    """A root whose `children` tokens (spread over the whole vocabulary, so
    over many chunks and CTAs) are all rejected: the draw removes every one."""
    B, N = 4, children + 1
    g = torch.Generator(device="cpu").manual_seed(8200 + children + V)
    x = (torch.randn((B, N, V), generator=g) * 3).to(torch.bfloat16)
    rng = np.random.default_rng(8200 + V)
    tok = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        row = x[b, 0].float().numpy()
        low = np.argsort(row, kind="stable")[: max(children * 20, V // 2)]
        tok[b, 1:] = rng.choice(low, size=children, replace=False)   # unlikely tokens, anywhere
    par = np.zeros((B, N), dtype=np.int32)
    par[:, 0] = -1
    u = np.full((B, N), 0.999, dtype=np.float32)
    xd = x.to(DEV)
    got = sv.spec_verify_tree(xd, torch.from_numpy(tok).to(DEV), torch.from_numpy(par).to(DEV), 1,
                              temperature=1.0, uniforms=torch.from_numpy(u).to(DEV), rule=sv.RULE_POWER,
                              alpha=0.3)
    ref = O.verify_tree(f64(xd), tok, par, 1, 1.0, u.astype(np.float64), rule=O.RULE_POWER, alpha=0.3)
    assert (ref["num_accepted"] == 0).all()
    compare(got, ref, stochastic=True)
    drawn = host(got["tokens"])[:, 0]
    for b in range(B):
        assert drawn[b] not in set(tok[b, 1:].tolist())


def test_many_requests_and_repeat_calls_are_identical():
    ti = W.eagle_tree(B=200, V=4096, seed=8300, device=DEV)
    run = lambda: sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth, temperature=1.0,
                                      uniforms=ti.uniforms, rule=sv.RULE_POWER, alpha=0.3)
    a, b = run(), run()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    ref = O.verify_tree(f64(ti.target), host(ti.node_tokens), host(ti.parents), ti.max_depth, 1.0,
                        f64(ti.uniforms), rule=O.RULE_POWER, alpha=0.3)
    compare(a, ref, stochastic=True, max_exempt=12)


@pytest.mark.parametrize("N,max_depth", [(1, 3), (2, 0), (5, 1), (700, 40)])
def test_tree_sizes_on_the_cluster_path(N, max_depth):
    """Random trees on the cluster path: a root alone (bonus draw from row 0),
    a depth cap of 0 (the root's children are never tested), and more nodes
    than the staged merge holds (700 rows: per-row serial merges)."""
    B, V = 3, 4096
    rng = np.random.default_rng(8500 + N)
    par = np.zeros((B, N), dtype=np.int32)
    par[:, 0] = -1
    for n in range(1, N):
        par[:, n] = rng.integers(0, n, size=B)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    tok[:, 0] = 0
    g = torch.Generator(device="cpu").manual_seed(8500 + N)
    x = (torch.randn((B, N, V), generator=g) * 3).to(torch.bfloat16).to(DEV)
    u = rng.random((B, N)).astype(np.float32)
    got = sv.spec_verify_tree(x, torch.from_numpy(tok).to(DEV), torch.from_numpy(par).to(DEV), max_depth,
                              temperature=1.0, uniforms=torch.from_numpy(u).to(DEV), rule=sv.RULE_POWER, alpha=0.3)
    ref = O.verify_tree(f64(x), tok, par, max_depth, 1.0, u.astype(np.float64), rule=O.RULE_POWER, alpha=0.3)
    compare(got, ref, stochastic=True)
    if max_depth == 0 and N > 1:
        assert (host(got["status"]) & sv.STATUS_DEPTH_EXCEEDED).all()
