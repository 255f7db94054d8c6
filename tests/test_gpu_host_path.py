"""spec_verify_greedy_host: greedy verification of logits in host memory,
streamed to the GPU in groups through two staging slots. Checked against the
device entry point on the same inputs (tokens, counts and status identical;
log-probabilities to float rounding) and against the oracle: several group
sizes (one request, an uneven last group, one group for all), padded host
rows (pitched copies), pageable and page-locked buffers, K = 0, and two calls
in a row on one workspace."""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import workloads as W
from oracle import spec_oracle as O
from parity_utils import compare, f64, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ATOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.load_library()


def _same_as_device(got, ci):
    ref = sv.spec_verify_greedy(ci.target, ci.draft_tokens)
    torch.cuda.synchronize()
    for k in ("tokens", "num_accepted", "status"):
        assert torch.equal(got[k], ref[k].cpu()), k
    for k in ("logprob", "mu"):
        assert np.allclose(got[k].numpy(), ref[k].cpu().numpy(), atol=ATOL, rtol=0), k


@pytest.mark.parametrize("dtype,V,group", [
    (torch.bfloat16, 4099, 0), (torch.bfloat16, 4099, 1), (torch.bfloat16, 4099, 3),
    (torch.float32, 32000, 8), (torch.float32, 32000, 5),
])
def test_host_path_matches_device_path_and_oracle(dtype, V, group):
    ci = W.greedy_chain(B=8, K=5, V=V, dtype=dtype, p_match=0.7, seed=8400 + V + group, device=DEV)
    xh = ci.target.cpu().pin_memory()
    dh = ci.draft_tokens.cpu().pin_memory()
    got = sv.spec_verify_greedy_host(xh, dh, group=group)
    _same_as_device(got, ci)
    compare(got, O.verify_greedy(f64(ci.target), host(ci.draft_tokens)))


def test_padded_host_rows_and_pageable_buffers():
    ci = W.greedy_chain(B=5, K=3, V=9001, dtype=torch.float32, p_match=0.8, seed=8410, device=DEV)
    B, R, V = ci.target.shape
    buf = torch.full((B, R, V + 7), float("nan"), dtype=torch.float32)     # pageable, pitch V + 7
    buf[:, :, :V] = ci.target.cpu()
    xh = buf[:, :, :V]
    assert xh.stride(1) == V + 7
    got = sv.spec_verify_greedy_host(xh, ci.draft_tokens.cpu(), group=2)
    _same_as_device(got, ci)
    compare(got, O.verify_greedy(f64(ci.target), host(ci.draft_tokens)))


def test_one_row_per_request():
    ci = W.greedy_chain(B=6, K=0, V=5000, dtype=torch.bfloat16, seed=8420, device=DEV)
    got = sv.spec_verify_greedy_host(ci.target.cpu(), ci.draft_tokens.cpu(), group=4)
    _same_as_device(got, ci)
    assert (got["num_accepted"] == 0).all()


def test_long_rows_many_groups_and_two_calls_on_one_workspace():
    # 4 requests of 256 rows of V = 50257 bf16 (25.7 MB each), one per group:
    # the slots are reused (groups 2 and 3 wait for groups 0 and 1)
    lib = sv.load_library()
    cis = [W.greedy_chain(B=4, K=255, V=50257, dtype=torch.bfloat16, p_match=0.97, seed=8430 + i, device=DEV)
           for i in range(2)]
    need = lib.spec_verify_greedy_host_workspace_size(4, 255, 50257, 1, 1)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    outs = []
    for ci in cis:
        got = sv.spec_verify_greedy_host(ci.target.cpu().pin_memory(), ci.draft_tokens.cpu().pin_memory(),
                                         group=1, workspace=ws)
        outs.append({k: v.clone() for k, v in got.items()})
    for got, ci in zip(outs, cis):
        _same_as_device(got, ci)
