"""GPU checks of early-exit greedy verification: tokens, num_accepted and
status identical to spec_verify_greedy (itself parity-tested against the
oracle) and log-probs equal within rounding (a row is summed by one CTA
here, by several there); parity with the oracle on the rows the decision
reads; bytes read between the oracle's bounds (oracle/early_exit.py); the
caller's state array back at zero."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import workloads as W
from oracle import early_exit as E
from oracle import spec_oracle as O
from parity_utils import compare, f64, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
KEYS = ("tokens", "num_accepted", "logprob", "mu", "status")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def _same(a, b):
    for k in ("tokens", "num_accepted", "status"):
        assert torch.equal(a[k], b[k]), k
    for k in ("logprob", "mu"):
        assert torch.allclose(a[k], b[k], atol=2e-5, rtol=0), k


def _bytes_ok(got, ci, es):
    B, R, V = ci.target.shape
    lo, hi = E.bytes_bounds(host(got["num_accepted"]), R - 1, V, es)
    br = int(host(got["bytes_read"])[0])
    assert lo <= br <= hi + B * R * 32, (lo, br, hi)   # each row read as its 16-byte hull
    return br, hi


def test_long_chain_reads_a_fraction_and_matches():
    B, K, Vv = 8, 4095, 50257
    ci = W.greedy_chain(B=B, K=K, V=Vv, dtype=torch.bfloat16, p_match=0.95, seed=7600, device=DEV)
    state = torch.zeros(2 * B, dtype=torch.int32, device=DEV)
    plain = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    for _ in range(2):                                   # the state is reused
        got = sv.spec_verify_greedy_early(ci.target, ci.draft_tokens, state=state)
        _same(got, plain)
        assert int(state.count_nonzero()) == 0
    br, hi = _bytes_ok(got, ci, 2)
    assert br < 0.25 * hi
    n = host(got["num_accepted"]).astype(np.int64)
    L = int(n.max() + 2)
    ref = O.verify_greedy(f64(ci.target[:, :L]), host(ci.draft_tokens[:, :L - 1]))
    assert np.array_equal(ref["num_accepted"], n)
    assert np.array_equal(host(got["tokens"])[:, :L], ref["tokens"][:, :L])


@pytest.mark.parametrize("B,K,Vv,dtype", [(32, 5, 128256, torch.bfloat16), (5, 300, 5003, torch.float32),
                                          (3, 0, 1000, torch.bfloat16), (6, 40, 7, torch.float32),
                                          (4, 64, 33, torch.bfloat16)])
def test_short_and_odd_shapes_match_the_oracle(B, K, Vv, dtype):
    ci = W.greedy_chain(B=B, K=K, V=Vv, dtype=dtype, p_match=0.9, seed=7601 + K, device=DEV)
    got = sv.spec_verify_greedy_early(ci.target, ci.draft_tokens)
    compare(got, O.verify_greedy(f64(ci.target), host(ci.draft_tokens)))
    _same(got, sv.spec_verify_greedy(ci.target, ci.draft_tokens))
    _bytes_ok(got, ci, 2 if dtype == torch.bfloat16 else 4)


def test_all_accepted_reads_everything():
    ci = W.greedy_chain(B=4, K=200, V=3000, dtype=torch.bfloat16, p_match=1.0, seed=7610, device=DEV)
    got = sv.spec_verify_greedy_early(ci.target, ci.draft_tokens)
    assert (host(got["num_accepted"]) == 200).all()
    br, hi = _bytes_ok(got, ci, 2)
    assert br >= hi


def test_padded_rows():
    x = W.greedy_chain(B=6, K=50, V=2001, dtype=torch.bfloat16, p_match=0.9, seed=7611, device=DEV)
    padded = torch.full((6, 51, 2001 + 5), float("-inf"), dtype=torch.bfloat16, device=DEV)
    padded[:, :, :2001] = x.target
    view = padded[:, :, :2001]
    got = sv.spec_verify_greedy_early(view, x.draft_tokens)
    compare(got, O.verify_greedy(f64(x.target), host(x.draft_tokens)))
