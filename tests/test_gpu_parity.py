"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs, at the workload sizes and at small and edge shapes.

Workloads (synthetic, shapes from the pages):
  toy          B=4, K=4, V=32 fp32, draft mix 0.8 p + 0.2 softmax(noise)
  llama chain  V=128256 bf16 N(0, 3^2), K=5, B in {1, 8, 32}, greedy
  qwen sample  V=151936 fp32, B=64, K=4, draft = target + N(0, 1), exact rule
  eagle tree   V=128256 bf16, B=32, 64 nodes, depth 5: greedy, power 0.3,
               relaxed 0.1
  long chain   V=50257 bf16, B=8, K+1=4096 rows, greedy (sampled: the oracle
               reads only the rows up to each request's decision)
"""

import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import verify as V
from speculative_decoding_verification_72_gb300 import workloads as W
from oracle import spec_oracle as O
from parity_utils import compare, f64, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def oracle_greedy(ci):
    return O.verify_greedy(f64(ci.target), host(ci.draft_tokens))


def oracle_sample(ci, rule=O.RULE_EXACT, tau=0.0, alpha=1.0, with_draft=True):
    y = f64(ci.draft_logits) if (with_draft and ci.draft_logits is not None) else None
    return O.verify_sample(f64(ci.target), y, host(ci.draft_tokens), ci.temperature,
                           f64(ci.uniforms), rule=rule, tau=tau, alpha=alpha)


def gpu_sample(ci, rule=O.RULE_EXACT, tau=0.0, alpha=1.0, with_draft=True):
    return sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms,
                                 draft_logits=ci.draft_logits if with_draft else None,
                                 temperature=ci.temperature, rule=rule, tau=tau, alpha=alpha)


# ----------------------------------------------------------------- toy config

def test_toy_greedy():
    ci = W.toy_chain(device=DEV)
    ci.draft_tokens = W.toy_greedy_drafts(ci.target)
    compare(sv.spec_verify_greedy(ci.target, ci.draft_tokens), oracle_greedy(ci))


@pytest.mark.parametrize("seed", [7200, 7201, 7202, 7203])
def test_toy_sample_exact(seed):
    ci = W.toy_chain(B=64, seed=seed, device=DEV)
    compare(gpu_sample(ci), oracle_sample(ci), stochastic=True)


@pytest.mark.parametrize("rule,tau,alpha", [(O.RULE_EXACT, 0.0, 1.0), (O.RULE_POWER, 0.0, 0.3),
                                            (O.RULE_RELAXED, 0.1, 1.0)])
def test_toy_sample_deterministic_drafts(rule, tau, alpha):
    ci = W.toy_chain(B=128, seed=7204, device=DEV)
    ci.draft_tokens = W.toy_greedy_drafts(ci.target, p_match=0.6, seed=3)
    compare(gpu_sample(ci, rule, tau, alpha, with_draft=False),
            oracle_sample(ci, rule, tau, alpha, with_draft=False), stochastic=True)


# ------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("B", [1, 8, 32])
def test_greedy_llama_vocab(B):
    ci = W.greedy_chain(B=B, K=5, V=128256, dtype=torch.bfloat16, seed=7201, device=DEV)
    compare(sv.spec_verify_greedy(ci.target, ci.draft_tokens), oracle_greedy(ci))


def test_stochastic_qwen_vocab():
    ci = W.stochastic_chain(B=64, K=4, V=151936, seed=7202, device=DEV)
    exempt = compare(gpu_sample(ci), oracle_sample(ci), stochastic=True)
    assert exempt <= 4


@pytest.mark.parametrize("mode", ["greedy", "power", "relaxed"])
def test_eagle_tree(mode):
    ti = W.eagle_tree(B=32, V=128256, seed=7203, device=DEV)
    x = f64(ti.target)
    tok, par = host(ti.node_tokens), host(ti.parents)
    if mode == "greedy":
        got = sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth)
        ref = O.verify_tree(x, tok, par, ti.max_depth, 0.0)
        compare(got, ref)
        return
    rule, tau, alpha = (O.RULE_POWER, 0.0, 0.3) if mode == "power" else (O.RULE_RELAXED, 0.1, 1.0)
    got = sv.spec_verify_tree(ti.target, ti.node_tokens, ti.parents, ti.max_depth,
                              temperature=1.0, uniforms=ti.uniforms, rule=rule, tau=tau, alpha=alpha)
    ref = O.verify_tree(x, tok, par, ti.max_depth, 1.0, f64(ti.uniforms), rule=rule, tau=tau,
                        alpha=alpha)
    assert compare(got, ref, stochastic=True) <= 2


def test_long_chain_sampled():
    B, K, Vv = 8, 4095, 50257
    ci = W.greedy_chain(B=B, K=K, V=Vv, dtype=torch.bfloat16, p_match=0.95, seed=7204, device=DEV)
    got = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    n_gpu = host(got["num_accepted"]).astype(np.int64)
    L = int(min(K + 1, n_gpu.max() + 2))
    ref = O.verify_greedy(f64(ci.target[:, :L]), host(ci.draft_tokens[:, : L - 1]))
    # the oracle on the first L rows reaches the same decision iff n < L - 1
    assert np.array_equal(ref["num_accepted"], n_gpu)
    tok = host(got["tokens"]).astype(np.int64)
    assert np.array_equal(tok[:, :L], ref["tokens"][:, :L])
    assert (tok[:, L:] == -1).all()
    assert np.allclose(host(got["logprob"])[:, :L], ref["logprob"][:, :L], atol=1e-4)
    assert (host(got["mu"])[:, L:] == 0).all() and (host(got["status"]) == 0).all()


# ----------------------------------------------------------- edge shapes

@pytest.mark.parametrize("B,K,Vv,dtype", [
    (1, 0, 7, torch.bfloat16), (3, 1, 1, torch.float32), (5, 2, 8, torch.bfloat16),
    (4, 3, 37, torch.bfloat16), (2, 4, 37, torch.float32), (3, 2, 16385, torch.bfloat16),
    (2, 1, 40001, torch.float32), (6, 7, 50257, torch.bfloat16), (2, 300, 513, torch.bfloat16)])
def test_greedy_edge_shapes(B, K, Vv, dtype):
    ci = W.greedy_chain(B=B, K=K, V=Vv, dtype=dtype, p_match=0.9, seed=B * 1000 + K, device=DEV)
    compare(sv.spec_verify_greedy(ci.target, ci.draft_tokens), oracle_greedy(ci))


@pytest.mark.parametrize("K", [255, 256, 600])
def test_greedy_decision_past_the_first_block(K):
    # p_match near 1 puts the first mismatch past the first 256-row block
    ci = W.greedy_chain(B=4, K=K, V=300, dtype=torch.bfloat16, p_match=0.998, seed=K, device=DEV)
    got = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    compare(got, oracle_greedy(ci))
    ci.uniforms = torch.zeros_like(ci.uniforms)     # u = 0 accepts every valid draft
    compare(gpu_sample(ci, with_draft=False), oracle_sample(ci, with_draft=False), stochastic=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("pad", [1, 3, 8])
def test_padded_row_stride(dtype, pad):
    B, K, Vv = 4, 3, 20011
    ci = W.greedy_chain(B=B, K=K, V=Vv, dtype=dtype, p_match=0.9, seed=pad, device=DEV)
    big = torch.zeros((B, K + 1, Vv + pad), dtype=dtype, device=DEV)
    big[:, :, :Vv] = ci.target
    view = big[:, :, :Vv]
    assert view.stride(1) == Vv + pad
    compare(sv.spec_verify_greedy(view, ci.draft_tokens), oracle_greedy(ci))


def test_ties_across_segments_take_lowest_index():
    B, K, Vv = 3, 2, 100003
    x = torch.randn((B, K + 1, Vv), device=DEV).mul(3).to(torch.bfloat16)
    x[0, 0, [90001, 70000, 20001, 5]] = 40.0   # equal maxima in different segments
    x[0, 1, [99999, 16063, 16064]] = 50.0
    x[1] = 1.0                                  # all equal: argmax 0
    x[2, :, [3, 4]] = 30.0
    d = torch.tensor([[5, 16063], [0, 0], [3, 4]], dtype=torch.int32, device=DEV)
    got = sv.spec_verify_greedy(x, d)
    ref = O.verify_greedy(f64(x), host(d))
    compare(got, ref)
    assert host(got["tokens"])[0, 0] == 5 and host(got["num_accepted"])[0] == 2


def test_masked_and_nonfinite_rows():
    B, K, Vv = 4, 2, 3001
    x = torch.randn((B, K + 1, Vv), device=DEV) * 3
    x[:, :, ::7] = -float("inf")
    x[1, 1, :] = -float("inf")           # fully masked row, read by the decision
    x[2, 2, :] = -float("inf")           # bonus row of request 2 fully masked
    x[3, 2, :] = -float("inf")           # after request 3's first mismatch: not read
    am = torch.argmax(x[:, :K], -1).to(torch.int32)
    d = am.clone()
    d[3, 0] = (d[3, 0] + 1) % Vv
    got = sv.spec_verify_greedy(x, d)
    ref = O.verify_greedy(f64(x), host(d))
    st = host(got["status"])
    assert st[1] & sv.STATUS_NONFINITE_ROW and st[2] & sv.STATUS_NONFINITE_ROW
    assert st[0] == 0 and st[3] == 0
    for b in (0, 3):
        assert np.array_equal(host(got["tokens"])[b], ref["tokens"][b])
        assert np.allclose(host(got["logprob"])[b], ref["logprob"][b], atol=1e-4)


def test_bad_tokens():
    ci = W.greedy_chain(B=4, K=3, V=999, dtype=torch.bfloat16, p_match=1.0, seed=5, device=DEV)
    d = ci.draft_tokens.clone()
    d[0, 1] = 999
    d[1, 0] = -7
    d[2, 2] = 1 << 30
    ci.draft_tokens = d
    got = sv.spec_verify_greedy(ci.target, d)
    compare(got, oracle_greedy(ci))
    assert (host(got["status"])[:3] == sv.STATUS_BAD_TOKEN).all()
    ci.uniforms = torch.zeros_like(ci.uniforms)
    compare(gpu_sample(ci, with_draft=False), oracle_sample(ci, with_draft=False), stochastic=True)


def test_zero_mass_draft_token():
    Vv = 64
    x = torch.randn((2, 2, Vv), device=DEV)
    y = torch.randn((2, 1, Vv), device=DEV)
    x[0, 0, 5] = -float("inf")
    y[0, 0, 5] = -float("inf")
    d = torch.tensor([[5], [int(torch.argmax(y[1, 0]))]], dtype=torch.int32, device=DEV)
    u = torch.rand((2, 2), device=DEV)
    ci = W.ChainInputs(target=x, draft_tokens=d, uniforms=u, draft_logits=y)
    got = gpu_sample(ci)
    ref = oracle_sample(ci)
    compare(got, ref, stochastic=True)
    assert host(got["status"])[0] == sv.STATUS_ZERO_MASS and host(got["num_accepted"])[0] == 0


def test_relaxed_extremes_and_temperature():
    ci = W.toy_chain(B=32, V=500, seed=9, device=DEV)
    ci.draft_tokens = W.toy_greedy_drafts(ci.target, p_match=0.5, seed=4)
    got = gpu_sample(ci, O.RULE_RELAXED, 0.0, 1.0, with_draft=False)
    assert (host(got["num_accepted"]) == 4).all()
    # tau = 0: any draft with p < 1e-5 counts as a near tie of p >= tau although
    # acceptance is certain (asserted above), so the exemption count is unbounded here
    compare(got, oracle_sample(ci, O.RULE_RELAXED, 0.0, 1.0, with_draft=False), stochastic=True,
            max_exempt=ci.target.shape[0])
    got = gpu_sample(ci, O.RULE_RELAXED, 1.5, 1.0, with_draft=False)
    assert (host(got["num_accepted"]) == 0).all()
    ci2 = W.stochastic_chain(B=16, K=3, V=5000, temperature=0.7, seed=12, device=DEV)
    compare(gpu_sample(ci2), oracle_sample(ci2), stochastic=True)
    ci3 = W.stochastic_chain(B=16, K=3, V=5000, dtype=torch.bfloat16, temperature=1.6, seed=13,
                             device=DEV)
    compare(gpu_sample(ci3), oracle_sample(ci3), stochastic=True)


def test_tree_bad_parents_and_depth_cap():
    ti = W.eagle_tree(B=6, V=3000, seed=21, device=DEV)
    par = ti.parents.clone()
    par[0, 9] = 9          # self link
    par[1, 0] = 0          # root link
    par[2, 20] = 63        # forward link
    tok = ti.node_tokens.clone()
    tok[3, 1] = -1
    for T, depth in ((0.0, 5), (0.0, 2), (1.0, 3)):
        got = sv.spec_verify_tree(ti.target, tok, par, depth, temperature=T, uniforms=ti.uniforms)
        ref = O.verify_tree(f64(ti.target), host(tok), host(par), depth, T,
                            None if T == 0 else f64(ti.uniforms))
        compare(got, ref, stochastic=T > 0)
        st = host(got["status"])
        assert (st[:3] & sv.STATUS_BAD_PARENT).all()


def test_exact_tree_and_chain_agree_on_chain_shaped_trees():
    B, K, Vv = 16, 6, 2000
    ci = W.greedy_chain(B=B, K=K, V=Vv, dtype=torch.float32, p_match=0.7, seed=31, device=DEV)
    par = torch.arange(-1, K, device=DEV, dtype=torch.int32).repeat(B, 1)
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device=DEV), ci.draft_tokens], 1)
    ut = torch.cat([ci.uniforms[:, K:], ci.uniforms[:, :K]], 1)
    for rule, tau, alpha in ((0, 0.0, 1.0), (2, 0.0, 0.3)):
        chain = gpu_sample(ci, rule, tau, alpha, with_draft=False)
        tree = sv.spec_verify_tree(ci.target, tok, par, K, temperature=1.0, uniforms=ut,
                                   rule=rule, tau=tau, alpha=alpha)
        ref = oracle_sample(ci, rule, tau, alpha, with_draft=False)
        compare(chain, ref, stochastic=True)
        compare(tree, ref, stochastic=True)


def test_repeat_calls_are_bit_identical():
    ci = W.stochastic_chain(B=32, K=4, V=151936, seed=77, device=DEV)
    a = gpu_sample(ci)
    b = gpu_sample(ci)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    g1 = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    g2 = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_outputs_stay_in_bounds():
    """Canary-padded output buffers through the raw C ABI."""
    lib = sv.load_library()
    B, K, Vv = 5, 4, 7001
    ci = W.greedy_chain(B=B, K=K, V=Vv, dtype=torch.bfloat16, seed=8, device=DEV)
    R, pad = K + 1, 64
    canary = -12345
    tok = torch.full((B * R + 2 * pad,), canary, dtype=torch.int32, device=DEV)
    num = torch.full((B + 2 * pad,), canary, dtype=torch.int32, device=DEV)
    lp = torch.full((B * R + 2 * pad,), -7.0, dtype=torch.float32, device=DEV)
    mu = torch.full((B * R + 2 * pad,), -7.0, dtype=torch.float32, device=DEV)
    st = torch.full((B + 2 * pad,), canary, dtype=torch.int32, device=DEV)
    need = lib.spec_verify_greedy_workspace_size(B, K, Vv, 1)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    P = ctypes.c_void_p
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.spec_verify_greedy(P(ci.target.data_ptr()), 1, Vv, P(ci.draft_tokens.data_ptr()), B, K,
                                Vv, P(tok.data_ptr() + 4 * pad), P(num.data_ptr() + 4 * pad),
                                P(lp.data_ptr() + 4 * pad), P(mu.data_ptr() + 4 * pad),
                                P(st.data_ptr() + 4 * pad), P(ws.data_ptr()), need, P(stream))
    assert rc == 0
    torch.cuda.synchronize()
    for t, c in ((tok, canary), (num, canary), (st, canary), (lp, -7.0), (mu, -7.0)):
        h = host(t)
        assert (h[:pad] == c).all() and (h[-pad:] == c).all()
    ref = oracle_greedy(ci)
    assert np.array_equal(host(tok)[pad:-pad].reshape(B, R), ref["tokens"])
