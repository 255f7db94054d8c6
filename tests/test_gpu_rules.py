"""GPU parity of the acceptance-rule options against the float64 oracle:
the relaxed rule's rank bound (top_k; rank = logits strictly greater than the
token's, raw logits) on chains and trees, and the power and relaxed rules with
draft logits, whose mu needs the extra pass over the emitted rows (nanospec
README, acceptance rules; spec-decode README for the residual).

Drafts for the rank tests are taken at a seeded rank r in [0, 2 top_k] of
their row, so both sides of the bound are hit; one case uses integer-valued
bf16 logits so that ranks are decided among many equal values.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def _ranked_drafts(target, K, max_rank, seed):
    """Draft i of request b = the token at a random rank r < max_rank of row i
    (descending, equal values in index order)."""
    B, V = target.shape[0], target.shape[-1]
    max_rank = min(max_rank, V)
    order = torch.argsort(target[:, :K].float(), dim=-1, descending=True, stable=True)
    g = torch.Generator(device=target.device).manual_seed(seed)
    r = torch.randint(0, max_rank, (B, K), generator=g, device=target.device)
    return torch.gather(order, -1, r.unsqueeze(-1)).squeeze(-1).to(torch.int32).contiguous()


def _uniforms(B, R, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.rand((B, R), generator=g, device=DEV, dtype=torch.float32)


def _sample_pair(x, drafts, u, y=None, T=1.0, rule=O.RULE_EXACT, tau=0.0, top_k=0, alpha=1.0):
    got = sv.spec_verify_sample(x, drafts, u, draft_logits=y, temperature=T, rule=rule, tau=tau,
                                top_k=top_k, alpha=alpha)
    ref = O.verify_sample(f64(x), None if y is None else f64(y), host(drafts), T, f64(u),
                          rule=rule, tau=tau, top_k=top_k, alpha=alpha)
    return got, ref


# ------------------------------------------- relaxed rank bound, chains

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [32, 1000, 70001])
@pytest.mark.parametrize("top_k,tau", [(1, 2.0), (3, 2.0), (16, 2.0), (4, 0.05)])
def test_relaxed_top_k_deterministic_drafts(dtype, V, top_k, tau):
    B, K = 48, 4
    x = W.greedy_chain(B=B, K=K, V=V, dtype=dtype, seed=7300 + V, device=DEV).target
    d = _ranked_drafts(x, K, 2 * top_k + 1, seed=V + top_k)
    u = _uniforms(B, K + 1, seed=11)
    got, ref = _sample_pair(x, d, u, rule=O.RULE_RELAXED, tau=tau, top_k=top_k)
    assert compare(got, ref, stochastic=True) <= 2


@pytest.mark.parametrize("top_k", [1, 2, 5, 16])
def test_relaxed_top_k_with_many_equal_logits(top_k):
    B, K, V = 64, 4, 300
    g = torch.Generator(device=DEV).manual_seed(7310 + top_k)
    x = torch.randint(-4, 5, (B, K + 1, V), generator=g, device=DEV).to(torch.bfloat16)
    d = _ranked_drafts(x, K, 3 * top_k + 3, seed=top_k)
    got, ref = _sample_pair(x, d, _uniforms(B, K + 1, 12), rule=O.RULE_RELAXED, tau=2.0, top_k=top_k)
    assert compare(got, ref, stochastic=True) <= 1
    # with tau out of reach the decision is the rank alone: exact, no near ties
    assert (host(got["num_accepted"]) == ref["num_accepted"]).all()


def test_top_k_at_least_the_vocabulary_accepts_everything():
    B, K, V = 16, 5, 8
    x = W.greedy_chain(B=B, K=K, V=V, dtype=torch.float32, seed=7320, device=DEV).target
    d = _ranked_drafts(x, K, V, seed=3)
    got, ref = _sample_pair(x, d, _uniforms(B, K + 1, 13), rule=O.RULE_RELAXED, tau=2.0, top_k=16)
    compare(got, ref, stochastic=True)
    assert (host(got["num_accepted"]) == K).all()


# --------------------------------------- power / relaxed with draft logits

@pytest.mark.parametrize("seed", [7330, 7331])
@pytest.mark.parametrize("rule,tau,top_k,alpha", [
    (O.RULE_POWER, 0.0, 0, 0.3), (O.RULE_POWER, 0.0, 0, 1.0), (O.RULE_POWER, 0.0, 0, 2.5),
    (O.RULE_RELAXED, 0.05, 0, 1.0), (O.RULE_RELAXED, 0.05, 3, 1.0), (O.RULE_RELAXED, 2.0, 1, 1.0)])
def test_toy_rules_with_draft_logits(seed, rule, tau, top_k, alpha):
    ci = W.toy_chain(B=128, seed=seed, device=DEV)
    got, ref = _sample_pair(ci.target, ci.draft_tokens, ci.uniforms, ci.draft_logits, 1.0,
                            rule, tau, top_k, alpha)
    assert compare(got, ref, stochastic=True) <= 3


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rule,tau,alpha", [(O.RULE_POWER, 0.0, 0.5), (O.RULE_RELAXED, 0.01, 1.0)])
def test_rules_with_draft_logits_several_chunks(dtype, rule, tau, alpha):
    # V = 20000 spans 5 vocabulary chunks of the mu pass, the last one ragged
    ci = W.stochastic_chain(B=24, K=4, V=20000, dtype=dtype, seed=7340, device=DEV)
    got, ref = _sample_pair(ci.target, ci.draft_tokens, ci.uniforms, ci.draft_logits, 1.0,
                            rule, tau, 0, alpha)
    assert compare(got, ref, stochastic=True) <= 2


def test_relaxed_top_k_with_draft_logits():
    # the oracle ranks every vocabulary entry one by one here, so V stays small
    ci = W.stochastic_chain(B=32, K=3, V=256, seed=7350, device=DEV)
    got, ref = _sample_pair(ci.target, ci.draft_tokens, ci.uniforms, ci.draft_logits, 1.0,
                            O.RULE_RELAXED, 0.2, 4, 1.0)
    assert compare(got, ref, stochastic=True) <= 2


def test_power_one_with_draft_logits_matches_the_exact_rule():
    ci = W.stochastic_chain(B=64, K=4, V=5000, seed=7360, device=DEV)
    a = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits)
    b = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits,
                              rule=O.RULE_POWER, alpha=1.0)
    n_a, n_b = host(a["num_accepted"]), host(b["num_accepted"])
    same = n_a == n_b    # a near tie may split them (the two compute acceptance differently)
    assert same.mean() > 0.95
    assert np.array_equal(host(a["tokens"])[same], host(b["tokens"])[same])
    assert np.allclose(host(a["mu"])[same], host(b["mu"])[same], atol=1e-4)


def test_power_rule_with_draft_logits_qwen_vocab():
    ci = W.stochastic_chain(B=64, K=4, V=151936, seed=7202, device=DEV)
    got, ref = _sample_pair(ci.target, ci.draft_tokens, ci.uniforms, ci.draft_logits, 1.0,
                            O.RULE_POWER, 0.0, 0, 0.5)
    assert compare(got, ref, stochastic=True) <= 4


# ------------------------------------------- relaxed rank bound, trees

@pytest.mark.parametrize("V,B,top_k,tau", [(20000, 8, 4, 0.1), (20000, 8, 2, 2.0), (128256, 32, 8, 0.1)])
def test_tree_relaxed_top_k(V, B, top_k, tau):
    ti = W.eagle_tree(B=B, V=V, seed=7370, device=DEV)
    got = sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth, temperature=1.0,
                              uniforms=ti.uniforms, rule=O.RULE_RELAXED, tau=tau, top_k=top_k)
    ref = O.verify_tree(f64(ti.target), host(ti.node_tokens), host(ti.parents), ti.max_depth, 1.0,
                        f64(ti.uniforms), rule=O.RULE_RELAXED, tau=tau, top_k=top_k)
    assert compare(got, ref, stochastic=True) <= 2
