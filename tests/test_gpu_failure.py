"""GPU tests of the failure paths the C ABI promises (include/spec_verify.h):

* a NaN inside a row the decision reads sets SV_STATUS_NONFINITE_ROW for that
  request only (chain rows 0..n, the tree path's rows, target and draft rows
  of a stochastic chain), while a NaN in a row the decision does not read
  changes nothing; the other requests match the oracle exactly. The oracle
  flags the same rows (row_is_finite), so status is compared bit for bit.
  Detection rests on the row pass's maximum ignoring NaN (max.bf16x2,
  max.f32) while the exponential sum turns NaN.
* a bounded wait that nothing completes gives up: spec_verify_selftest_wait
  runs the same bounded mbarrier wait the streaming kernels use on a phase no
  copy or thread completes, reports SV_STATUS_TIMEOUT, and the context stays
  usable for the next verification call.
"""

import time

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import workloads as W
from oracle import spec_oracle as O
from parity_utils import compare, f64, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
NAN = float("nan")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def _non_argmax(row, rng):
    """A vocabulary index that is not the row's argmax (so the NaN cannot
    change which token wins)."""
    am = int(torch.argmax(row.float()).item())
    j = int(rng.integers(0, row.numel() - 1))
    return j + (j >= am)


def _status(got):
    return host(got["status"]).astype(np.int64)


def test_nan_in_read_chain_rows_is_flagged_per_request():
    ci = W.greedy_chain(B=8, K=5, V=128256, dtype=torch.bfloat16, p_match=0.7, seed=901, device=DEV)
    clean = O.verify_greedy(f64(ci.target), host(ci.draft_tokens))
    n = clean["num_accepted"]
    rng = np.random.default_rng(5)
    read_rows = {0: 0, 1: int(n[1])}                 # row 0, and the last row request 1's decision reads
    unread = [b for b in range(8) if b not in read_rows and n[b] < 5]
    assert unread, "the seed leaves a request that rejects before its last row"
    b_unread = unread[0]
    poisoned = dict(read_rows)
    poisoned[b_unread] = int(n[b_unread]) + 1        # after the decision: not read
    for b, r in poisoned.items():
        ci.target[b, r, _non_argmax(ci.target[b, r], rng)] = NAN
    got = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    ref = O.verify_greedy(f64(ci.target), host(ci.draft_tokens))
    torch.cuda.synchronize()
    st = _status(got)
    for b in read_rows:
        assert st[b] & sv.STATUS_NONFINITE_ROW, (b, st[b])
        assert ref["status"][b] & O.STATUS_NONFINITE_ROW
    assert not (st[b_unread] & sv.STATUS_NONFINITE_ROW)
    # every request whose read rows are clean matches the oracle bit for bit
    keep = [b for b in range(8) if b not in read_rows]
    sub = {k: (v[keep] if isinstance(v, np.ndarray) else v) for k, v in ref.items()}
    compare({k: v[keep] for k, v in got.items()}, sub)


def test_nan_in_tree_path_row_is_flagged():
    ti = W.eagle_tree(B=8, V=128256, dtype=torch.bfloat16, seed=902, device=DEV)
    rng = np.random.default_rng(6)
    clean = O.verify_tree(f64(ti.target), host(ti.node_tokens), host(ti.parents), ti.max_depth, 0.0)
    # request 0: the root row (always on the path); request 1: a node off its path
    ti.target[0, 0, _non_argmax(ti.target[0, 0], rng)] = NAN
    path1 = set(int(v) for v in clean["nodes"][1] if v >= 0)
    off = [n for n in range(1, 64) if n not in path1]
    ti.target[1, off[0], _non_argmax(ti.target[1, off[0]], rng)] = NAN
    got = sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth)
    ref = O.verify_tree(f64(ti.target), host(ti.node_tokens), host(ti.parents), ti.max_depth, 0.0)
    torch.cuda.synchronize()
    st = _status(got)
    assert st[0] & sv.STATUS_NONFINITE_ROW and ref["status"][0] & O.STATUS_NONFINITE_ROW
    assert not (st[1] & sv.STATUS_NONFINITE_ROW)
    keep = list(range(1, 8))
    compare({k: v[keep] for k, v in got.items()},
            {k: (v[keep] if isinstance(v, np.ndarray) else v) for k, v in ref.items()})


def test_nan_in_stochastic_target_and_draft_rows_is_flagged():
    ci = W.stochastic_chain(B=8, K=4, V=151936, dtype=torch.float32, seed=903, device=DEV)
    rng = np.random.default_rng(7)
    ci.target[0, 0, _non_argmax(ci.target[0, 0], rng)] = NAN        # target row 0: always read
    ci.draft_logits[1, 0, _non_argmax(ci.draft_logits[1, 0], rng)] = NAN   # draft row 0: always read
    got = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits)
    ref = O.verify_sample(f64(ci.target), f64(ci.draft_logits), host(ci.draft_tokens), 1.0, f64(ci.uniforms))
    torch.cuda.synchronize()
    st = _status(got)
    for b in (0, 1):
        assert st[b] & sv.STATUS_NONFINITE_ROW, (b, st[b])
        assert ref["status"][b] & O.STATUS_NONFINITE_ROW
    keep = list(range(2, 8))
    compare({k: v[keep] for k, v in got.items()},
            {k: (v[keep] if isinstance(v, np.ndarray) else v) for k, v in ref.items()}, stochastic=True)


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = sv.spec_verify_selftest_wait()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(st.item()) == sv.STATUS_TIMEOUT
    assert sv.spec_verify_check_status(st) == sv.SV_ERR_TIMEOUT
    assert 0.015 <= waited < 5.0, waited          # about 20 ms of polling, never unbounded
    # the next call on the same context and stream works and matches the oracle
    ci = W.greedy_chain(B=4, K=5, V=4099, dtype=torch.bfloat16, seed=904, device=DEV)
    got = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    compare(got, O.verify_greedy(f64(ci.target), host(ci.draft_tokens)))
    assert sv.spec_verify_check_status(got["status"]) == 0
