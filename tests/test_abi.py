"""C-ABI checks that need no GPU: the library loads, exports every function
include/spec_verify.h declares, and rejects invalid arguments on the host
with the documented codes before launching anything."""

import ctypes
import os
import re

import pytest

import speculative_decoding_verification_72_gb300 as sv
from speculative_decoding_verification_72_gb300 import verify as V

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED_DTYPE = 0, 1, 2
SV_ERR_WORKSPACE_TOO_SMALL, SV_ERR_NOT_SUPPORTED, SV_ERR_TIMEOUT = 3, 5, 6
FAKE = 0x10000          # 64 KB-aligned stand-in for a device pointer; never dereferenced


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(sv.library_path()):
        from speculative_decoding_verification_72_gb300 import build
        build.build()
    return sv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("spec_verify_greedy", "spec_verify_sample", "spec_verify_tree",
              "spec_verify_greedy_ex", "spec_verify_sample_ex", "spec_verify_tree_ex",
              "spec_verify_status_string", "spec_verify_abi_version", "spec_verify_workspace_size",
              "spec_verify_check_status", "spec_verify_selftest_wait"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in V._SIGS, f"binding lacks a signature for {name}"


def test_abi_version_and_status_strings(lib):
    assert lib.spec_verify_abi_version() == 3
    for code in range(7):
        s = lib.spec_verify_status_string(code).decode()
        assert s and "unknown" not in s
    assert "unknown" in lib.spec_verify_status_string(99).decode()


def test_workspace_sizes(lib):
    g = lib.spec_verify_greedy_workspace_size(32, 5, 128256, 1)
    assert g >= 32 * 6 * 16 and g % 256 == 0
    assert lib.spec_verify_sample_workspace_size(64, 4, 151936, 0, 1) > \
        lib.spec_verify_sample_workspace_size(64, 4, 151936, 0, 0)
    assert lib.spec_verify_tree_workspace_size(32, 64, 128256, 1) > 0
    assert lib.spec_verify_greedy_workspace_size(4, 5, 0, 1) == 0      # V < 1
    assert lib.spec_verify_greedy_workspace_size(4, 5, 100, 7) == 0    # dtype
    assert lib.spec_verify_tree_workspace_size(4, 2000, 100, 1) == 0   # N too large
    assert lib.spec_verify_greedy_workspace_size(0, 5, 100, 1) > 0


def test_one_workspace_size_serves_every_verification_call(lib):
    for B, R, Vv, dt in ((32, 6, 128256, 1), (64, 5, 151936, 0), (32, 64, 128256, 1), (8, 4096, 50257, 1),
                         (1, 1, 7, 0), (0, 6, 100, 1)):
        one = lib.spec_verify_workspace_size(B, R, Vv, dt)
        assert one > 0 and one % 256 == 0
        assert one >= lib.spec_verify_greedy_workspace_size(B, R - 1, Vv, dt)
        assert one >= lib.spec_verify_sample_workspace_size(B, R - 1, Vv, dt, 1)
        assert one >= lib.spec_verify_sample_workspace_size(B, R - 1, Vv, dt, 0)
        if R <= 1024:
            assert one >= lib.spec_verify_tree_workspace_size(B, R, Vv, dt)
        # and it is the largest of them, not more
        needs = [lib.spec_verify_greedy_workspace_size(B, R - 1, Vv, dt),
                 lib.spec_verify_sample_workspace_size(B, R - 1, Vv, dt, 1),
                 lib.spec_verify_sample_workspace_size(B, R - 1, Vv, dt, 0)]
        if R <= 1024:
            needs.append(lib.spec_verify_tree_workspace_size(B, R, Vv, dt))
        assert one == max(needs)
    assert lib.spec_verify_workspace_size(4, 0, 100, 1) == 0      # rows_per_req < 1
    assert lib.spec_verify_workspace_size(-1, 6, 100, 1) == 0
    assert lib.spec_verify_workspace_size(4, 6, 0, 1) == 0
    assert lib.spec_verify_workspace_size(4, 6, 100, 5) == 0      # dtype


def test_check_status_turns_the_timeout_bit_into_a_return_code(lib):
    arr = (ctypes.c_int32 * 4)(0, 4, 64, 128)
    assert lib.spec_verify_check_status(arr, 4) == SV_OK            # per-request outcomes, not errors
    arr[2] = 64 | 32
    assert lib.spec_verify_check_status(arr, 4) == SV_ERR_TIMEOUT
    assert lib.spec_verify_check_status(arr, 2) == SV_OK            # only the first B are read
    assert lib.spec_verify_check_status(None, 0) == SV_OK
    assert lib.spec_verify_check_status(None, 3) == SV_ERR_INVALID_ARG
    assert lib.spec_verify_check_status(arr, -1) == SV_ERR_INVALID_ARG
    assert "TIMEOUT" in lib.spec_verify_status_string(SV_ERR_TIMEOUT).decode()


def test_selftest_rejects_bad_pointers(lib):
    assert lib.spec_verify_selftest_wait(None, None) == SV_ERR_INVALID_ARG
    assert lib.spec_verify_selftest_wait(ctypes.c_void_p(FAKE + 2), None) == SV_ERR_INVALID_ARG


def test_status_bits_match_the_header():
    text = open(HEADER).read()
    for name, val in (("SV_STATUS_BAD_TOKEN", V.STATUS_BAD_TOKEN), ("SV_STATUS_BAD_PARENT", V.STATUS_BAD_PARENT),
                      ("SV_STATUS_NONFINITE_ROW", V.STATUS_NONFINITE_ROW), ("SV_STATUS_ZERO_MASS", V.STATUS_ZERO_MASS),
                      ("SV_STATUS_DEPTH_EXCEEDED", V.STATUS_DEPTH_EXCEEDED), ("SV_STATUS_TIMEOUT", V.STATUS_TIMEOUT),
                      ("SV_STATUS_STOPPED", V.STATUS_STOPPED), ("SV_STATUS_CAPPED", V.STATUS_CAPPED),
                      ("SV_STATUS_BAD_PAGE", V.STATUS_BAD_PAGE), ("SV_ERR_TIMEOUT", V.SV_ERR_TIMEOUT)):
        m = re.search(r"#define\s+" + name + r"\s+(\d+)", text)
        assert m and int(m.group(1)) == val, name


def test_kernels_take_status_bits_from_the_header():
    """No kernel source spells a status bit as a number: each names the
    header's constant, so kernels and ABI cannot drift apart."""
    csrc = os.path.join(ROOT, "speculative_decoding_verification_72_gb300", "csrc")
    pat = re.compile(r"(status\w*\s*(\|=|=)\s*[1-9])|(\bst\s*\|=\s*[1-9])|(stat\s*\|=\s*[1-9])|"
                     r"(atomicOr\(&s_status,\s*[1-9])|(\?\s*(4|32)\s*:\s*0)")
    for name in os.listdir(csrc):
        if name.endswith((".cu", ".cuh")):
            for i, line in enumerate(open(os.path.join(csrc, name)), 1):
                code = line.split("//")[0]
                assert not pat.search(code), f"{name}:{i}: literal status bit: {line.strip()}"


def _greedy(lib, **kw):
    a = dict(x=FAKE, dtype=1, stride=100, d=FAKE, B=2, K=3, V=100,
             tok=FAKE, num=FAKE, lp=FAKE, mu=FAKE, st=FAKE, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.spec_verify_greedy(P(a["x"]), a["dtype"], a["stride"], P(a["d"]), a["B"], a["K"],
                                  a["V"], P(a["tok"]), P(a["num"]), P(a["lp"]), P(a["mu"]),
                                  P(a["st"]), P(a["ws"]), a["wsb"], P(0))


def test_greedy_host_validation(lib):
    assert _greedy(lib, dtype=3) == SV_ERR_UNSUPPORTED_DTYPE
    assert _greedy(lib, V=0) == SV_ERR_INVALID_ARG
    assert _greedy(lib, K=-1) == SV_ERR_INVALID_ARG
    assert _greedy(lib, stride=99) == SV_ERR_INVALID_ARG
    assert _greedy(lib, x=0) == SV_ERR_INVALID_ARG
    assert _greedy(lib, d=0) == SV_ERR_INVALID_ARG
    assert _greedy(lib, tok=0) == SV_ERR_INVALID_ARG
    assert _greedy(lib, ws=0) == SV_ERR_INVALID_ARG
    assert _greedy(lib, x=FAKE + 1) == SV_ERR_INVALID_ARG          # misaligned bf16
    assert _greedy(lib, ws=FAKE + 8) == SV_ERR_INVALID_ARG         # workspace not 16-byte aligned
    assert _greedy(lib, wsb=16) == SV_ERR_WORKSPACE_TOO_SMALL
    assert _greedy(lib, B=0, x=0, d=0, tok=0, num=0, ws=0) == SV_OK  # nothing to do


def _greedy_host(lib, **kw):
    a = dict(x=FAKE, dtype=1, stride=100, d=FAKE, B=2, K=3, V=100, group=0,
             tok=FAKE, num=FAKE, lp=FAKE, mu=FAKE, st=FAKE, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.spec_verify_greedy_host(P(a["x"]), a["dtype"], a["stride"], P(a["d"]), a["B"], a["K"],
                                       a["V"], a["group"], P(a["tok"]), P(a["num"]), P(a["lp"]), P(a["mu"]),
                                       P(a["st"]), P(a["ws"]), a["wsb"], P(0))


def test_greedy_host_path_sizes_and_validation(lib):
    one = lib.spec_verify_greedy_host_workspace_size
    B, K, Vv = 8, 4095, 50257                        # 411.7 MB of bf16 logits per request
    req = (K + 1) * Vv * 2
    w_auto = one(B, K, Vv, 1, 0)                     # 256 MB groups: one request each
    assert w_auto == one(B, K, Vv, 1, 1)
    assert 2 * req <= w_auto < 2 * req + lib.spec_verify_greedy_workspace_size(1, K, Vv, 1) + (1 << 20)
    assert one(B, K, Vv, 1, 3) >= 2 * 3 * req        # two staging slots of 3 requests
    assert one(B, K, Vv, 1, 100) == one(B, K, Vv, 1, B)   # a group never exceeds B
    small = one(32, 5, 128256, 1, 0)                 # 32 requests fit one 256 MB group
    assert small >= 2 * 32 * 6 * 128256 * 2 and small % 256 == 0
    assert one(4, 5, 0, 1, 0) == 0 and one(4, 5, 100, 7, 0) == 0 and one(4, 5, 100, 1, -1) == 0
    assert one(-1, 5, 100, 1, 0) == 0
    assert _greedy_host(lib, dtype=3) == SV_ERR_UNSUPPORTED_DTYPE
    assert _greedy_host(lib, V=0) == SV_ERR_INVALID_ARG
    assert _greedy_host(lib, stride=99) == SV_ERR_INVALID_ARG
    assert _greedy_host(lib, group=-2) == SV_ERR_INVALID_ARG
    assert _greedy_host(lib, x=0) == SV_ERR_INVALID_ARG
    assert _greedy_host(lib, d=0) == SV_ERR_INVALID_ARG
    assert _greedy_host(lib, num=0) == SV_ERR_INVALID_ARG
    assert _greedy_host(lib, ws=FAKE + 16) == SV_ERR_INVALID_ARG   # staging wants 256-byte alignment
    assert _greedy_host(lib, wsb=4096) == SV_ERR_WORKSPACE_TOO_SMALL
    assert _greedy_host(lib, B=0, x=0, d=0, tok=0, num=0, ws=0) == SV_OK


def _sample(lib, rule=(0, 0.0, 0, 1.0), T=1.0, draft=FAKE, **kw):
    a = dict(x=FAKE, dtype=0, stride=100, d=FAKE, B=2, K=3, V=100, u=FAKE, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.spec_verify_sample(P(a["x"]), a["dtype"], a["stride"], P(draft), 100, P(a["d"]),
                                  a["B"], a["K"], a["V"], T, P(a["u"]), V.RuleParams(*rule),
                                  P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                  P(a["ws"]), a["wsb"], P(0))


def test_sample_host_validation(lib):
    assert _sample(lib, T=0.0) == SV_ERR_INVALID_ARG
    assert _sample(lib, T=float("nan")) == SV_ERR_INVALID_ARG
    assert _sample(lib, T=float("inf")) == SV_ERR_INVALID_ARG
    assert _sample(lib, u=0) == SV_ERR_INVALID_ARG
    assert _sample(lib, rule=(7, 0.0, 0, 1.0)) == SV_ERR_INVALID_ARG
    assert _sample(lib, rule=(2, 0.0, 0, 0.0), draft=0) == SV_ERR_INVALID_ARG     # alpha <= 0
    assert _sample(lib, rule=(1, float("nan"), 0, 1.0), draft=0) == SV_ERR_INVALID_ARG
    assert _sample(lib, rule=(1, 0.1, 99, 1.0), draft=0) == SV_ERR_INVALID_ARG    # top_k > max
    # valid rule combinations pass validation and stop at the workspace check
    assert _sample(lib, rule=(1, 0.1, 2, 1.0), draft=0, wsb=64) == SV_ERR_WORKSPACE_TOO_SMALL
    assert _sample(lib, rule=(1, 0.1, 16, 1.0), wsb=64) == SV_ERR_WORKSPACE_TOO_SMALL
    assert _sample(lib, rule=(2, 0.0, 0, 0.3), wsb=64) == SV_ERR_WORKSPACE_TOO_SMALL  # power with q
    assert _sample(lib, wsb=64) == SV_ERR_WORKSPACE_TOO_SMALL


def _tree(lib, T=0.0, **kw):
    a = dict(x=FAKE, dtype=1, stride=100, tok=FAKE, par=FAKE, B=2, N=8, V=100, depth=5,
             u=FAKE, nodes=FAKE, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.spec_verify_tree(P(a["x"]), a["dtype"], a["stride"], P(a["tok"]), P(a["par"]),
                                a["B"], a["N"], a["V"], a["depth"], T, P(a["u"]),
                                V.RuleParams(0, 0.0, 0, 1.0),
                                P(FAKE), P(a["nodes"]), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                P(a["ws"]), a["wsb"], P(0))


def test_tree_host_validation(lib):
    assert _tree(lib, N=0) == SV_ERR_INVALID_ARG
    assert _tree(lib, N=1025) == SV_ERR_INVALID_ARG
    assert _tree(lib, depth=-1) == SV_ERR_INVALID_ARG
    assert _tree(lib, par=0) == SV_ERR_INVALID_ARG
    assert _tree(lib, nodes=0) == SV_ERR_INVALID_ARG
    assert _tree(lib, T=0.5, u=0) == SV_ERR_INVALID_ARG
    assert _tree(lib, T=-1.0) == SV_ERR_INVALID_ARG
    assert _tree(lib, wsb=32) == SV_ERR_WORKSPACE_TOO_SMALL


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros((1, 2, 8))
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_greedy(x, torch.zeros((1, 1), dtype=torch.int32))


def _greedy_ex(lib, fin, **kw):
    a = dict(x=FAKE, dtype=1, stride=100, d=FAKE, B=2, K=3, V=100, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.spec_verify_greedy_ex(P(a["x"]), a["dtype"], a["stride"], P(a["d"]), a["B"], a["K"], a["V"],
                                     P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                     ctypes.byref(fin) if fin is not None else None,
                                     P(a["ws"]), a["wsb"], P(0))


def test_finish_params_validation(lib):
    F = V.FinishParams
    # out_len missing, n_stop out of range, stop ids missing, misaligned pointers
    assert _greedy_ex(lib, F(None, 0, None, None, None)) == SV_ERR_INVALID_ARG
    assert _greedy_ex(lib, F(FAKE, 17, None, FAKE, None)) == SV_ERR_INVALID_ARG
    assert _greedy_ex(lib, F(FAKE, -1, None, FAKE, None)) == SV_ERR_INVALID_ARG
    assert _greedy_ex(lib, F(None, 2, None, FAKE, None)) == SV_ERR_INVALID_ARG
    assert _greedy_ex(lib, F(FAKE + 2, 1, None, FAKE, None)) == SV_ERR_INVALID_ARG
    assert _greedy_ex(lib, F(FAKE, 1, None, FAKE, FAKE + 4)) == SV_ERR_INVALID_ARG
    # valid parameters reach the workspace check; no finish behaves like the plain call
    assert _greedy_ex(lib, F(FAKE, 2, FAKE, FAKE, FAKE), wsb=16) == SV_ERR_WORKSPACE_TOO_SMALL
    assert _greedy_ex(lib, None, wsb=16) == SV_ERR_WORKSPACE_TOO_SMALL
    assert _greedy_ex(lib, F(FAKE, 2, None, FAKE, None), B=0) == SV_OK
