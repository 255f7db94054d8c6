"""spec_verify_greedy_static: the entry point for callers that cannot
allocate device memory (they are handed fixed input and output buffers and
no allocator, or must not allocate once serving has started). It takes no
workspace; its scratch is the library's static device array.

Checked through the raw C ABI against spec_verify_greedy with a caller
workspace, on two calls in a row with different inputs. The static array
keeps the previous call's contents, so the larger call runs first: the
second, smaller call then reads its partials from an array still holding
the first call's (more) partials, and must ignore them. Plus the size
limit. This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SV_BF16 = 1
SV_ERR_WORKSPACE_TOO_SMALL = 3
ATOL = 1e-4
MAX_STATIC_ROWS = 33353           # rows that fit the 4 MiB static scratch array
P = ctypes.c_void_p


def _outs(B, R, dev):
    return (torch.full((B, R), -7, dtype=torch.int32, device=dev),
            torch.full((B,), -7, dtype=torch.int32, device=dev),
            torch.full((B, R), -7.0, dtype=torch.float32, device=dev),
            torch.full((B, R), -7.0, dtype=torch.float32, device=dev),
            torch.full((B,), -7, dtype=torch.int32, device=dev))


def _call(lib, ci, outs, static, ws=None):
    B, R, V = ci.target.shape
    stream = P(torch.cuda.current_stream().cuda_stream)
    args = [P(ci.target.data_ptr()), SV_BF16, V, P(ci.draft_tokens.data_ptr()), B, R - 1, V]
    args += [P(t.data_ptr()) for t in outs]
    if static:
        return lib.spec_verify_greedy_static(*args, stream)
    return lib.spec_verify_greedy(*args, P(ws.data_ptr()), ws.numel(), stream)


def test_static_scratch_matches_workspace_path_on_two_calls():
    assert torch.cuda.is_available()
    lib = sv.load_library()
    dev = torch.device("cuda:0")
    # larger call first (2408 rows + one partial per CTA), then a smaller one
    # (192 rows) over the leftovers
    for seed, (B, K, V) in ((12, (8, 300, 50257)), (11, (32, 5, 128256))):
        ci = W.greedy_chain(B=B, K=K, V=V, dtype=torch.bfloat16, p_match=0.9, seed=seed, device=dev)
        need = lib.spec_verify_greedy_workspace_size(B, K, V, SV_BF16)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        ref = _outs(B, K + 1, dev)
        got = _outs(B, K + 1, dev)
        assert _call(lib, ci, ref, static=False, ws=ws) == 0
        assert _call(lib, ci, got, static=True) == 0
        torch.cuda.synchronize()
        for k in (0, 1, 4):                      # tokens, num_accepted, status
            assert torch.equal(got[k], ref[k])
        for k in (2, 3):                         # logprob, mu
            assert np.allclose(got[k].cpu().numpy(), ref[k].cpu().numpy(), atol=ATOL, rtol=0)
        assert (got[1] >= 0).all()


def test_static_scratch_rejects_requests_beyond_its_size():
    lib = sv.load_library()
    dev = torch.device("cuda:0")
    B, K, V = 1, MAX_STATIC_ROWS, 8           # MAX_STATIC_ROWS + 1 rows
    x = torch.zeros((B, K + 1, V), dtype=torch.bfloat16, device=dev)
    d = torch.zeros((B, K), dtype=torch.int32, device=dev)
    outs = _outs(B, K + 1, dev)
    ci = W.ChainInputs(target=x, draft_tokens=d, uniforms=torch.zeros((B, K + 1), device=dev))
    assert _call(lib, ci, outs, static=True) == SV_ERR_WORKSPACE_TOO_SMALL
    # the largest request that fits is accepted
    x2 = torch.zeros((B, MAX_STATIC_ROWS, V), dtype=torch.bfloat16, device=dev)
    d2 = torch.zeros((B, MAX_STATIC_ROWS - 1), dtype=torch.int32, device=dev)
    outs2 = _outs(B, MAX_STATIC_ROWS, dev)
    ci2 = W.ChainInputs(target=x2, draft_tokens=d2, uniforms=torch.zeros((B, 1), device=dev))
    assert _call(lib, ci2, outs2, static=True) == 0
    torch.cuda.synchronize()
    assert int(outs2[1][0]) == MAX_STATIC_ROWS - 1   # all-zero rows: every draft 0 is the argmax
