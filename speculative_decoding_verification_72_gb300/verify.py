"""Thin ctypes binding of libspecverify (include/spec_verify.h).

Argument marshalling only: every step of verification runs in the library's
CUDA kernels. Tensors are torch CUDA tensors; outputs and the workspace are
allocated here with torch (device memory plumbing) and the call is enqueued
on the current torch stream of the input's device. There is no CPU fallback:
a missing library or a CPU tensor raises SpecVerifyError.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

SV_OK = 0
SV_F32 = 0
SV_BF16 = 1

RULE_EXACT = 0
RULE_RELAXED = 1
RULE_POWER = 2

STATUS_BAD_TOKEN = 1
STATUS_BAD_PARENT = 2
STATUS_NONFINITE_ROW = 4
STATUS_ZERO_MASS = 8
STATUS_DEPTH_EXCEEDED = 16
STATUS_TIMEOUT = 32
STATUS_STOPPED = 64
STATUS_CAPPED = 128
STATUS_BAD_PAGE = 256

SV_ERR_TIMEOUT = 6

_LIB = None
_LOCK = threading.Lock()
_WS = {}


class SpecVerifyError(RuntimeError):
    pass


class RuleParams(ctypes.Structure):
    _fields_ = [("rule", ctypes.c_int32), ("tau", ctypes.c_float),
                ("top_k", ctypes.c_int32), ("alpha", ctypes.c_float)]


class FinishParams(ctypes.Structure):
    _fields_ = [("stop_ids", ctypes.c_void_p), ("n_stop", ctypes.c_int32),
                ("max_new", ctypes.c_void_p), ("out_len", ctypes.c_void_p),
                ("counters", ctypes.c_void_p)]


def library_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libspecverify.so")


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGS = {
    "spec_verify_abi_version": (_I32, []),
    "spec_verify_status_string": (ctypes.c_char_p, [_I32]),
    "spec_verify_greedy_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "spec_verify_sample_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "spec_verify_tree_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "spec_verify_greedy": (_I32, [_P, _I32, _I64, _P, _I32, _I32, _I32,
                                  _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_sample": (_I32, [_P, _I32, _I64, _P, _I64, _P, _I32, _I32, _I32,
                                  _F, _P, RuleParams,
                                  _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_tree": (_I32, [_P, _I32, _I64, _P, _P, _I32, _I32, _I32, _I32,
                                _F, _P, RuleParams,
                                _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_greedy_static": (_I32, [_P, _I32, _I64, _P, _I32, _I32, _I32,
                                         _P, _P, _P, _P, _P, _P]),
    "spec_verify_greedy_host_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "spec_verify_greedy_host": (_I32, [_P, _I32, _I64, _P, _I32, _I32, _I32, _I32,
                                       _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_greedy_early": (_I32, [_P, _I32, _I64, _P, _I32, _I32, _I32,
                                        _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_tree_build_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "spec_verify_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "spec_verify_check_status": (_I32, [_P, _I32]),
    "spec_verify_selftest_wait": (_I32, [_P, _P]),
    "spec_tree_build": (_I32, [_P, _I32, _I64, _I32, _I32, _I32, _I32, _I32, _F,
                               _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_kv_compact": (_I32, [_P, _I64, _I32, _P, _I32, _I32, _P, _P, _I32, _P, _I32, _I32, _P, _P, _P]),
    "spec_verify_greedy_ex": (_I32, [_P, _I32, _I64, _P, _I32, _I32, _I32,
                                     _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_sample_ex": (_I32, [_P, _I32, _I64, _P, _I64, _P, _I32, _I32, _I32,
                                     _F, _P, RuleParams,
                                     _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_verify_tree_ex": (_I32, [_P, _I32, _I64, _P, _P, _I32, _I32, _I32, _I32,
                                   _F, _P, RuleParams,
                                   _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
}


def load_library(path=None):
    """Load libspecverify.so (built in-tree by __graft_entry__.build())."""
    global _LIB
    with _LOCK:
        if _LIB is not None and path is None:
            return _LIB
        p = path or library_path()
        if not os.path.exists(p):
            raise SpecVerifyError(
                f"libspecverify.so is not built at {p}; run __graft_entry__.build() first")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _LIB = lib
        return lib


def _check(rc):
    if rc != SV_OK:
        msg = load_library().spec_verify_status_string(rc).decode()
        raise SpecVerifyError(f"libspecverify returned {rc}: {msg}")


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise SpecVerifyError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _rows_view(t, name):
    """(tensor, row_stride) for a [B, R, V] logits tensor whose rows are evenly
    strided (unit stride along V); otherwise a contiguous copy."""
    if t.dim() != 3:
        raise SpecVerifyError(f"{name} must be [B, rows, V]")
    if not t.is_cuda:
        raise SpecVerifyError(f"{name} must be a CUDA tensor")
    B, R, V = t.shape
    if t.stride(2) != 1 and V > 1:
        t = t.contiguous()
    if R > 1:
        rs, ok = t.stride(1), (B == 1 or t.stride(0) == R * t.stride(1))
    elif B > 1:
        rs, ok = t.stride(0), True
    else:
        rs, ok = V, True
    if not ok or rs < V:
        t = t.contiguous()
        rs = V
    return t, rs


def _i32(t, name, shape, device):
    """int32 contiguous copy on `device`; shape None = any 1-D length."""
    if not isinstance(t, torch.Tensor):
        t = torch.as_tensor(t, dtype=torch.int64)
    if shape is None:
        shape = (t.numel(),)
        t = t.reshape(-1)
    if tuple(t.shape) != tuple(shape):
        raise SpecVerifyError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.to(device=device, dtype=torch.int32).contiguous()


def _f32(t, name, shape, device):
    if not isinstance(t, torch.Tensor):
        t = torch.as_tensor(t)
    if tuple(t.shape) != tuple(shape):
        raise SpecVerifyError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.to(device=device, dtype=torch.float32).contiguous()


def _workspace(nbytes, device, stream):
    key = (device.index, stream)
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _WS[key] = ws
    return ws


def _ws(workspace, need, dev, stream):
    if workspace is None:
        return _workspace(need, dev, stream)
    if workspace.numel() * workspace.element_size() < need or not workspace.is_cuda:
        raise SpecVerifyError(f"workspace must be a CUDA tensor of at least {need} bytes")
    return workspace


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _outputs(B, cols, device, want_nodes=False, out=None):
    """Fresh output tensors, or the caller's (checked) when `out` is given."""
    if out is not None:
        need = {"tokens": (B, cols), "num_accepted": (B,), "logprob": (B, cols),
                "mu": (B, cols), "status": (B,)}
        if want_nodes:
            need["nodes"] = (B, cols)
        for k, shp in need.items():
            t = out.get(k)
            if t is None or tuple(t.shape) != shp or not t.is_contiguous() or t.device != device:
                raise SpecVerifyError(f"out[{k!r}] must be a contiguous {shp} tensor on {device}")
        return out
    out = dict(
        tokens=torch.empty((B, cols), dtype=torch.int32, device=device),
        num_accepted=torch.empty((B,), dtype=torch.int32, device=device),
        logprob=torch.empty((B, cols), dtype=torch.float32, device=device),
        mu=torch.empty((B, cols), dtype=torch.float32, device=device),
        status=torch.empty((B,), dtype=torch.int32, device=device),
    )
    if want_nodes:
        out["nodes"] = torch.empty((B, cols), dtype=torch.int32, device=device)
    return out


def _rule(rule, tau, top_k, alpha):
    return RuleParams(int(rule), float(tau), int(top_k), float(alpha))


def _finish(B, dev, out, stop_ids, max_new, counters):
    """(FinishParams pointer, tensors kept alive) when a finish option is
    given, else (None, None). Adds out["out_len"]."""
    if stop_ids is None and max_new is None and counters is None:
        return None, None
    stop = _i32(stop_ids if stop_ids is not None else [], "stop_ids", None, dev)
    cap = _i32(max_new, "max_new", (B,), dev) if max_new is not None else None
    if counters is not None:
        if (not isinstance(counters, torch.Tensor) or counters.dtype != torch.int64 or
                tuple(counters.shape) != (B, 4) or not counters.is_contiguous() or counters.device != dev):
            raise SpecVerifyError(f"counters must be a contiguous int64 ({B}, 4) tensor on {dev}")
    if out.get("out_len") is None:
        out["out_len"] = torch.empty((B,), dtype=torch.int32, device=dev)
    fp = FinishParams(_ptr(stop) if stop.numel() else None, int(stop.numel()),
                      _ptr(cap) if cap is not None else None, _ptr(out["out_len"]),
                      _ptr(counters) if counters is not None else None)
    return ctypes.byref(fp), (fp, stop, cap)


def spec_verify_greedy(target_logits, draft_tokens, workspace=None, out=None,
                       stop_ids=None, max_new=None, counters=None):
    """Greedy chain verification. target_logits [B, K+1, V] (bf16 / fp32,
    CUDA), draft_tokens [B, K]. Returns a dict of CUDA tensors: tokens,
    num_accepted, logprob, mu, status (the caller's `out` dict if given;
    with `out` and `workspace` given the call allocates nothing and can be
    captured in a CUDA graph). stop_ids / max_new [B] / counters (int64
    [B, 4], updated in place) select the finish step of include/spec_verify.h
    and add out["out_len"]."""
    lib = load_library()
    x, stride = _rows_view(target_logits, "target_logits")
    B, R, V = x.shape
    K = R - 1
    dev = x.device
    d = _i32(draft_tokens, "draft_tokens", (B, K), dev)
    out = _outputs(B, R, dev, out=out)
    stream = torch.cuda.current_stream(dev).cuda_stream
    need = lib.spec_verify_greedy_workspace_size(B, K, V, _dtype_code(x))
    if need == 0 and B > 0:
        raise SpecVerifyError("invalid sizes")
    ws = _ws(workspace, need, dev, stream)
    fin, _keep = _finish(B, dev, out, stop_ids, max_new, counters)
    rc = lib.spec_verify_greedy_ex(_ptr(x), _dtype_code(x), stride, _ptr(d), B, K, V,
                                   _ptr(out["tokens"]), _ptr(out["num_accepted"]),
                                   _ptr(out["logprob"]), _ptr(out["mu"]), _ptr(out["status"]), fin,
                                   _ptr(ws), ws.numel() * ws.element_size(), ctypes.c_void_p(stream))
    _check(rc)
    return out


def spec_verify_greedy_host(target_logits, draft_tokens, group=0, device=None, workspace=None, out=None):
    """Greedy chain verification of host-resident logits (spec_verify_greedy_host
    in include/spec_verify.h): target_logits [B, K+1, V] (bf16 / fp32) and
    draft_tokens [B, K] are CPU tensors (pinned for full copy speed); the
    call streams groups of `group` requests (0: the library's choice) to
    `device` (default: the current CUDA device) and returns CPU tensors
    tokens, num_accepted, logprob, mu, status (the caller's `out` dict of
    contiguous CPU tensors if given), valid once the current stream has
    completed (the function synchronizes it before returning)."""
    lib = load_library()
    if target_logits.dim() != 3 or target_logits.is_cuda:
        raise SpecVerifyError("target_logits must be a [B, rows, V] CPU tensor")
    x = target_logits
    if x.stride(2) != 1 or (x.shape[0] > 1 and x.stride(0) != x.shape[1] * x.stride(1)) or x.stride(1) < x.shape[2]:
        x = x.contiguous()
    B, R, V = x.shape
    K = R - 1
    stride = x.stride(1) if R > 1 else (x.stride(0) if B > 1 else V)
    d = draft_tokens
    if d.is_cuda or d.dtype != torch.int32 or tuple(d.shape) != (B, K) or not d.is_contiguous():
        raise SpecVerifyError(f"draft_tokens must be a contiguous int32 ({B}, {K}) CPU tensor")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if out is None:
        out = _outputs(B, R, torch.device("cpu"))
    else:
        for k, shp in {"tokens": (B, R), "num_accepted": (B,), "logprob": (B, R), "mu": (B, R),
                       "status": (B,)}.items():
            t = out.get(k)
            if t is None or tuple(t.shape) != shp or not t.is_contiguous() or t.is_cuda:
                raise SpecVerifyError(f"out[{k!r}] must be a contiguous {shp} CPU tensor")
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        need = lib.spec_verify_greedy_host_workspace_size(B, K, V, _dtype_code(x), int(group))
        if need == 0 and B > 0:
            raise SpecVerifyError("invalid sizes")
        ws = _ws(workspace, need, dev, stream)
        rc = lib.spec_verify_greedy_host(_ptr(x), _dtype_code(x), stride, _ptr(d), B, K, V, int(group),
                                         _ptr(out["tokens"]), _ptr(out["num_accepted"]),
                                         _ptr(out["logprob"]), _ptr(out["mu"]), _ptr(out["status"]),
                                         _ptr(ws), ws.numel() * ws.element_size(), ctypes.c_void_p(stream))
        _check(rc)
        torch.cuda.current_stream(dev).synchronize()
    return out


def spec_verify_sample(target_logits, draft_tokens, uniforms, draft_logits=None,
                       temperature=1.0, rule=RULE_EXACT, tau=0.0, top_k=0, alpha=1.0,
                       workspace=None, out=None, stop_ids=None, max_new=None, counters=None):
    """Stochastic chain verification (see include/spec_verify.h); finish
    options as for spec_verify_greedy."""
    lib = load_library()
    x, stride = _rows_view(target_logits, "target_logits")
    B, R, V = x.shape
    K = R - 1
    dev = x.device
    y, dstride = (None, 0)
    if draft_logits is not None:
        if draft_logits.dtype != x.dtype:
            raise SpecVerifyError("draft_logits must have the target's dtype")
        y, dstride = _rows_view(draft_logits, "draft_logits")
        if tuple(y.shape) != (B, K, V):
            raise SpecVerifyError(f"draft_logits must be {(B, K, V)}")
    d = _i32(draft_tokens, "draft_tokens", (B, K), dev)
    u = _f32(uniforms, "uniforms", (B, R), dev)
    out = _outputs(B, R, dev, out=out)
    stream = torch.cuda.current_stream(dev).cuda_stream
    need = lib.spec_verify_sample_workspace_size(B, K, V, _dtype_code(x), int(y is not None))
    ws = _ws(workspace, need, dev, stream)
    fin, _keep = _finish(B, dev, out, stop_ids, max_new, counters)
    rc = lib.spec_verify_sample_ex(_ptr(x), _dtype_code(x), stride, _ptr(y), dstride, _ptr(d),
                                   B, K, V, float(temperature), _ptr(u),
                                   _rule(rule, tau, top_k, alpha),
                                   _ptr(out["tokens"]), _ptr(out["num_accepted"]),
                                   _ptr(out["logprob"]), _ptr(out["mu"]), _ptr(out["status"]), fin,
                                   _ptr(ws), ws.numel() * ws.element_size(), ctypes.c_void_p(stream))
    _check(rc)
    return out


def spec_verify_tree(target_logits, node_tokens, parents, max_depth, temperature=0.0,
                     uniforms=None, rule=RULE_EXACT, tau=0.0, top_k=0, alpha=1.0,
                     workspace=None, out=None, stop_ids=None, max_new=None, counters=None):
    """Tree verification (see include/spec_verify.h). temperature 0 = greedy;
    finish options as for spec_verify_greedy."""
    lib = load_library()
    x, stride = _rows_view(target_logits, "target_logits")
    B, N, V = x.shape
    dev = x.device
    tok = _i32(node_tokens, "node_tokens", (B, N), dev)
    par = _i32(parents, "parents", (B, N), dev)
    u = None
    if float(temperature) != 0.0:
        u = _f32(uniforms, "uniforms", (B, N), dev)
    W = int(max_depth) + 1
    out = _outputs(B, W, dev, want_nodes=True, out=out)
    stream = torch.cuda.current_stream(dev).cuda_stream
    need = lib.spec_verify_tree_workspace_size(B, N, V, _dtype_code(x))
    if need == 0 and B > 0:
        raise SpecVerifyError("invalid sizes")
    ws = _ws(workspace, need, dev, stream)
    fin, _keep = _finish(B, dev, out, stop_ids, max_new, counters)
    rc = lib.spec_verify_tree_ex(_ptr(x), _dtype_code(x), stride, _ptr(tok), _ptr(par), B, N, V,
                                 int(max_depth), float(temperature), _ptr(u),
                                 _rule(rule, tau, top_k, alpha),
                                 _ptr(out["tokens"]), _ptr(out["nodes"]), _ptr(out["num_accepted"]),
                                 _ptr(out["logprob"]), _ptr(out["mu"]), _ptr(out["status"]), fin,
                                 _ptr(ws), ws.numel() * ws.element_size(), ctypes.c_void_p(stream))
    _check(rc)
    return out


_EARLY_STATE = {}


def spec_verify_greedy_early(target_logits, draft_tokens, state=None, workspace=None, out=None):
    """Early-exit greedy chain verification (include/spec_verify.h): the same
    outputs as spec_verify_greedy, plus out["bytes_read"] (int64 [1], logit
    bytes the call read). `state` is the caller's zero-filled int32 [2B]
    request state (left zero after each call); by default one cached per
    device, stream and B is used."""
    lib = load_library()
    x, stride = _rows_view(target_logits, "target_logits")
    B, R, V = x.shape
    K = R - 1
    dev = x.device
    d = _i32(draft_tokens, "draft_tokens", (B, K), dev)
    out = _outputs(B, R, dev, out=out)
    if out.get("bytes_read") is None:
        out["bytes_read"] = torch.zeros((1,), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    if state is None:
        key = (dev.index, stream, B)
        state = _EARLY_STATE.get(key)
        if state is None:
            state = _EARLY_STATE[key] = torch.zeros((2 * B,), dtype=torch.int32, device=dev)
    elif (state.dtype != torch.int32 or tuple(state.shape) != (2 * B,) or not state.is_contiguous() or
          state.device != dev):
        raise SpecVerifyError(f"state must be a contiguous int32 ({2 * B},) tensor on {dev}")
    need = lib.spec_verify_greedy_workspace_size(B, K, V, _dtype_code(x))
    if need == 0 and B > 0:
        raise SpecVerifyError("invalid sizes")
    ws = _ws(workspace, need, dev, stream)
    rc = lib.spec_verify_greedy_early(_ptr(x), _dtype_code(x), stride, _ptr(d), B, K, V,
                                      _ptr(out["tokens"]), _ptr(out["num_accepted"]),
                                      _ptr(out["logprob"]), _ptr(out["mu"]), _ptr(out["status"]),
                                      _ptr(state), _ptr(out["bytes_read"]),
                                      _ptr(ws), ws.numel() * ws.element_size(), ctypes.c_void_p(stream))
    _check(rc)
    return out


def spec_tree_build(draft_logits, depth, topk, n_nodes, temperature=1.0, workspace=None, out=None):
    """EAGLE-style draft tree from rank-ordered draft rows (include/spec_verify.h).
    draft_logits [B, 1 + (depth - 1) * topk, V]. Returns a dict of CUDA
    tensors: tokens, parents, scores [B, n_nodes] and status [B]; tokens and
    parents feed spec_verify_tree."""
    lib = load_library()
    x, stride = _rows_view(draft_logits, "draft_logits")
    B, R, V = x.shape
    if R != 1 + (int(depth) - 1) * int(topk):
        raise SpecVerifyError(f"draft_logits must have 1 + (depth - 1) * topk = {1 + (depth - 1) * topk} rows")
    dev = x.device
    if out is None:
        out = dict(tokens=torch.empty((B, n_nodes), dtype=torch.int32, device=dev),
                   parents=torch.empty((B, n_nodes), dtype=torch.int32, device=dev),
                   scores=torch.empty((B, n_nodes), dtype=torch.float32, device=dev),
                   status=torch.empty((B,), dtype=torch.int32, device=dev))
    stream = torch.cuda.current_stream(dev).cuda_stream
    need = lib.spec_tree_build_workspace_size(B, int(depth), int(topk), V)
    if need == 0 and B > 0:
        raise SpecVerifyError("invalid sizes")
    ws = _ws(workspace, need, dev, stream)
    rc = lib.spec_tree_build(_ptr(x), _dtype_code(x), stride, B, V, int(depth), int(topk), int(n_nodes),
                             float(temperature), _ptr(out["tokens"]), _ptr(out["parents"]),
                             _ptr(out["scores"]), _ptr(out["status"]),
                             _ptr(ws), ws.numel() * ws.element_size(), ctypes.c_void_p(stream))
    _check(rc)
    return out


def spec_kv_compact(kv, page_table, seq_base, path_nodes, num_accepted, max_nodes, out=None):
    """Move each request's accepted tree path into consecutive cache positions
    (include/spec_verify.h). kv [pages, page_size, ...] CUDA tensor (modified
    in place; each token row 16-byte multiple), page_table [B, max_pages],
    seq_base [B], path_nodes [B, cols] (out_nodes of spec_verify_tree),
    num_accepted [B]. Returns dict(out_len [B], status [B])."""
    lib = load_library()
    if not kv.is_cuda or kv.dim() < 3 or not kv.is_contiguous():
        raise SpecVerifyError("kv must be a contiguous CUDA tensor [pages, page_size, ...]")
    dev = kv.device
    pages, P = kv.shape[0], kv.shape[1]
    row_bytes = kv[0, 0].numel() * kv.element_size()
    B = page_table.shape[0]
    pt = _i32(page_table, "page_table", tuple(page_table.shape), dev)
    sb = _i32(seq_base, "seq_base", (B,), dev)
    pn = _i32(path_nodes, "path_nodes", tuple(path_nodes.shape), dev)
    na = _i32(num_accepted, "num_accepted", (B,), dev)
    if out is None:
        out = dict(out_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   status=torch.empty((B,), dtype=torch.int32, device=dev))
    stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.spec_kv_compact(_ptr(kv), row_bytes, row_bytes, _ptr(pt), pt.shape[1], P, _ptr(sb), _ptr(pn),
                             pn.shape[1], _ptr(na), B, int(max_nodes), _ptr(out["out_len"]), _ptr(out["status"]),
                             ctypes.c_void_p(stream))
    _check(rc)
    return out


def spec_verify_workspace_size(B, rows_per_req, V, dtype):
    """Workspace bytes that serve every verification entry point for B
    requests of rows_per_req target rows of V logits (include/spec_verify.h);
    dtype is torch.float32 or torch.bfloat16."""
    code = SV_F32 if dtype == torch.float32 else SV_BF16 if dtype == torch.bfloat16 else None
    if code is None:
        raise SpecVerifyError(f"dtype must be float32 or bfloat16, got {dtype}")
    need = load_library().spec_verify_workspace_size(int(B), int(rows_per_req), int(V), code)
    if need == 0:
        raise SpecVerifyError("invalid sizes")
    return need


def spec_verify_check_status(status):
    """SV_OK, or SV_ERR_TIMEOUT if any request's status has STATUS_TIMEOUT
    (status: int32 tensor, copied to the host)."""
    h = status.detach().to("cpu", torch.int32).contiguous()
    return load_library().spec_verify_check_status(_ptr(h), int(h.numel()))


def spec_verify_selftest_wait(device=None):
    """Runs the library's bounded-wait self-test on `device` (default: the
    current CUDA device) and returns the int32 status it wrote (device
    tensor [1]): STATUS_TIMEOUT when the wait gave up as designed."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if dev.type != "cuda":
        raise SpecVerifyError("the self-test needs a CUDA device")
    out = torch.full((1,), -1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(load_library().spec_verify_selftest_wait(_ptr(out), ctypes.c_void_p(stream)))
    return out
