"""GPU parity of the draw's less common paths against the float64 oracle:
logits whose buffers start off a 16-byte boundary (chunk copies clipped at
the buffer's ends, elements read from global memory), target and draft rows
at different alignments (element-by-element sums), more requests per CTA
than the CTA caches (descriptors and exclusion lists read from global
memory), masked draws with more rejected tokens in one chunk than a stage
descriptor carries, or more than are cached per request, and rows with more
chunks than the pick kernel keeps in shared memory."""

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


def _offset_view(x, off, pad):
    """x [B, R, V] copied into a flat buffer at element offset `off` with row
    pitch V + pad; returns the [B, R, V] strided view."""
    B, R, V = x.shape
    pitch = V + pad
    buf = torch.full((off + B * R * pitch + 8,), float("nan"), dtype=x.dtype, device=x.device)
    view = buf[off: off + B * R * pitch].view(B, R, pitch)[:, :, :V]
    view.copy_(x)
    assert view.stride(1) == pitch and view.data_ptr() % 16 == (off * x.element_size()) % 16
    return view


def _oracle_sample(ci, with_draft=True, rule=O.RULE_EXACT, alpha=1.0):
    y = f64(ci.draft_logits) if with_draft else None
    return O.verify_sample(f64(ci.target), y, host(ci.draft_tokens), ci.temperature, f64(ci.uniforms),
                           rule=rule, alpha=alpha)


@pytest.mark.parametrize("dtype,V,t_off,t_pad,d_off,d_pad", [
    (torch.float32, 9001, 1, 3, 3, 1),       # fp32: 3 chunks, target and draft at different phases
    (torch.float32, 9001, 2, 2, 2, 2),       # same phase, both starts off the boundary
    (torch.bfloat16, 20011, 5, 2, 2, 6),     # bf16: 3 chunks, different phases
    (torch.bfloat16, 20011, 3, 0, 3, 0),     # odd pitch, same phase
])
def test_residual_draws_with_unaligned_rows(dtype, V, t_off, t_pad, d_off, d_pad):
    ci = W.stochastic_chain(B=6, K=3, V=V, dtype=dtype, seed=7900 + V + t_off, device=DEV)
    tv = _offset_view(ci.target, t_off, t_pad)
    dv = _offset_view(ci.draft_logits, d_off, d_pad)
    got = sv.spec_verify_sample(tv, ci.draft_tokens, ci.uniforms, draft_logits=dv, temperature=ci.temperature)
    compare(got, _oracle_sample(ci), stochastic=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_masked_and_bonus_draws_with_unaligned_rows(dtype):
    ci = W.stochastic_chain(B=8, K=3, V=12007, dtype=dtype, seed=7910, device=DEV)
    tv = _offset_view(ci.target, 3, 5)
    got = sv.spec_verify_sample(tv, ci.draft_tokens, ci.uniforms, temperature=ci.temperature,
                                rule=sv.RULE_POWER, alpha=0.5)
    compare(got, _oracle_sample(ci, with_draft=False, rule=O.RULE_POWER, alpha=0.5), stochastic=True)


def test_more_requests_per_cta_than_it_caches():
    # V = 40: one chunk per request, so a chain call of 2600 requests gives
    # each of the ~304 chunk-sum CTAs 8-9 requests (more than the 8 it caches)
    ci = W.stochastic_chain(B=2600, K=2, V=40, seed=7920, device=DEV)
    got = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits,
                                temperature=ci.temperature)
    compare(got, _oracle_sample(ci), stochastic=True)
    got = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, temperature=ci.temperature,
                                rule=sv.RULE_POWER, alpha=0.3)
    compare(got, _oracle_sample(ci, with_draft=False, rule=O.RULE_POWER, alpha=0.3), stochastic=True)


@pytest.mark.parametrize("children,V", [(10, 300), (70, 300), (70, 20000)])
def test_wide_root_with_every_child_rejected(children, V):
    """A root with `children` low-probability children, all rejected: the
    draw removes them all (more than a stage descriptor holds; for 70, more
    than are cached per request)."""
    B, N = 4, children + 1
    g = torch.Generator(device="cpu").manual_seed(7930 + children + V)
    x = (torch.randn((B, N, V), generator=g) * 3).to(torch.bfloat16)
    tok = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        order = np.argsort(x[b, 0].float().numpy(), kind="stable")
        tok[b, 1:] = order[:children]       # the root row's least likely tokens
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


def test_more_chunks_than_the_pick_stages():
    # fp32 V = 1.2M: 293 chunks of 4096, past the 256 chunk sums the pick
    # kernel keeps in shared memory
    ci = W.stochastic_chain(B=3, K=1, V=1_200_000, seed=7940, device=DEV)
    got = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits,
                                temperature=ci.temperature)
    compare(got, _oracle_sample(ci), stochastic=True)
    ci.uniforms[:, 0] = 0.999999          # reject the draft: residual draws over all chunks
    got = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits,
                                temperature=ci.temperature)
    compare(got, _oracle_sample(ci), stochastic=True)


def test_exact_rule_chains_past_the_fused_length():
    # K + 1 > 16: the stochastic exact rule with draft logits runs the decide
    # kernel (the chunk-sum kernel decides only chains of up to 16 rows)
    ci = W.stochastic_chain(B=16, K=20, V=5000, seed=7950, device=DEV)
    got = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits,
                                temperature=ci.temperature)
    compare(got, _oracle_sample(ci), stochastic=True)
    # and the fused length itself (K + 1 = 16)
    ci = W.stochastic_chain(B=16, K=15, V=5000, seed=7951, device=DEV)
    got = sv.spec_verify_sample(ci.target, ci.draft_tokens, ci.uniforms, draft_logits=ci.draft_logits,
                                temperature=ci.temperature)
    compare(got, _oracle_sample(ci), stochastic=True)
