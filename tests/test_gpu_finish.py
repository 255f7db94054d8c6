"""GPU parity of the finish step (stop-set and max-new-tokens truncation,
per-request counters) against oracle/finish.py applied to the oracle's
verification, for every kernel that can end a call: the greedy chain and
greedy tree decide kernels, the draw kernel (stochastic chains and trees) and
the mu pass (power / relaxed with draft logits)."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import workloads as W
from oracle import finish as F
from oracle import spec_oracle as O
from parity_utils import compare, f64, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def _finish_inputs(ref, seed, width):
    """Stop ids taken from tokens the oracle emits (so some requests stop),
    random caps around the emitted length, and non-zero starting counters."""
    rng = np.random.default_rng(seed)
    tok = ref["tokens"]
    B = tok.shape[0]
    emitted = [int(t) for b in range(B) for t in tok[b, 1:int(ref["num_accepted"][b]) + 1]]
    stop = list(rng.choice(emitted, size=min(3, len(emitted)), replace=False)) if emitted else [0]
    stop.append(int(tok[0, 0]))
    max_new = rng.integers(-1, width + 2, size=B)
    counters = rng.integers(0, 50, size=(B, 4))
    return [int(s) for s in stop], max_new, counters


def _check(got, ref, stop, max_new, cnt0, offered, stochastic):
    ref_f, out_len, cnt = F.finish(ref, stop_ids=stop, max_new=max_new, counters=cnt0, offered=offered)
    compare(got, ref_f, stochastic=stochastic)
    exact = np.ones(len(out_len), dtype=bool)
    if stochastic:
        exact = ref["tie_pos"] < 0
    got_len = host(got["out_len"]).astype(np.int64)
    got_cnt = host(got["counters"]).astype(np.int64)
    assert np.array_equal(got_len[exact], out_len[exact])
    assert np.array_equal(got_cnt[exact], cnt[exact])
    assert exact.mean() > 0.9
    assert ((F.STATUS_STOPPED & host(got["status"])) != 0).any()     # the stop set was exercised
    assert ((F.STATUS_CAPPED & host(got["status"])) != 0).any()      # and the cap


def _run(fn, ref, seed, width, offered, stochastic=False):
    stop, max_new, cnt0 = _finish_inputs(ref, seed, width)
    counters = torch.tensor(cnt0, dtype=torch.int64, device=DEV)
    got = fn(stop_ids=stop, max_new=torch.tensor(max_new, dtype=torch.int32, device=DEV), counters=counters)
    got["counters"] = counters
    _check(got, ref, stop, max_new, cnt0, offered, stochastic)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_greedy_chain_finish(dtype):
    ci = W.greedy_chain(B=64, K=5, V=20000, dtype=dtype, p_match=0.85, seed=7500, device=DEV)
    ref = O.verify_greedy(f64(ci.target), host(ci.draft_tokens))
    _run(lambda **kw: sv.spec_verify_greedy(ci.target, ci.draft_tokens, **kw), ref, 1, 6, 5)


def test_greedy_tree_finish():
    ti = W.eagle_tree(B=32, V=20000, seed=7501, device=DEV)
    ref = O.verify_tree(f64(ti.target), host(ti.node_tokens), host(ti.parents), ti.max_depth, 0.0)
    _run(lambda **kw: sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth, **kw),
         ref, 2, ti.max_depth + 1, ti.max_depth)


def test_stochastic_chain_finish_after_the_draw():
    ci = W.toy_chain(B=256, seed=7502, device=DEV)
    ref = O.verify_sample(f64(ci.target), f64(ci.draft_logits), host(ci.draft_tokens), 1.0, f64(ci.uniforms))
    _run(lambda **kw: sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms,
                                            draft_logits=ci.draft_logits, **kw),
         ref, 3, 5, 4, stochastic=True)


def test_deterministic_draft_chain_finish():
    ci = W.toy_chain(B=256, seed=7503, device=DEV)
    d = W.toy_greedy_drafts(ci.target, p_match=0.7, seed=5)
    ref = O.verify_sample(f64(ci.target), None, host(d), 1.0, f64(ci.uniforms), rule=O.RULE_POWER, alpha=0.5)
    _run(lambda **kw: sv.spec_verify_sample(ci.target, d, ci.uniforms, rule=O.RULE_POWER, alpha=0.5, **kw),
         ref, 4, 5, 4, stochastic=True)


def test_power_rule_with_draft_logits_finish_after_the_mu_pass():
    ci = W.toy_chain(B=256, seed=7504, device=DEV)
    ref = O.verify_sample(f64(ci.target), f64(ci.draft_logits), host(ci.draft_tokens), 1.0, f64(ci.uniforms),
                          rule=O.RULE_POWER, alpha=0.4)
    _run(lambda **kw: sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms,
                                            draft_logits=ci.draft_logits, rule=O.RULE_POWER, alpha=0.4, **kw),
         ref, 5, 5, 4, stochastic=True)


def test_stochastic_tree_finish():
    ti = W.eagle_tree(B=32, V=20000, seed=7505, device=DEV)
    ref = O.verify_tree(f64(ti.target), host(ti.node_tokens), host(ti.parents), ti.max_depth, 1.0,
                        f64(ti.uniforms), rule=O.RULE_RELAXED, tau=0.05)
    _run(lambda **kw: sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth, 1.0,
                                          ti.uniforms, rule=O.RULE_RELAXED, tau=0.05, **kw),
         ref, 6, ti.max_depth + 1, ti.max_depth, stochastic=True)


def test_counters_accumulate_over_calls_and_plain_calls_are_unchanged():
    ci = W.greedy_chain(B=16, K=4, V=5000, dtype=torch.bfloat16, seed=7506, device=DEV)
    plain = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    counters = torch.zeros((16, 4), dtype=torch.int64, device=DEV)
    for _ in range(3):
        got = sv.spec_verify_greedy(ci.target, ci.draft_tokens, counters=counters)
    n = host(plain["num_accepted"]).astype(np.int64)
    c = host(counters)
    assert (c[:, 0] == 3).all() and (c[:, 1] == 12).all()
    assert np.array_equal(c[:, 2], 3 * n) and np.array_equal(c[:, 3], 3 * (n + 1))
    for k in ("tokens", "num_accepted", "logprob", "mu", "status"):   # no stop set, no cap: nothing cut
        assert torch.equal(got[k], plain[k])
    assert np.array_equal(host(got["out_len"]), n + 1)
