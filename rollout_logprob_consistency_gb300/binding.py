"""Thin ctypes binding over libtim.so (argument marshalling only).

Every step of the scoring and comparison runs in the CUDA library; this module
only checks tensor dtypes/devices, passes raw device pointers and sizes through
the C ABI declared in include/tim.h, and converts the status codes to
exceptions.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if libtim.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtim.so")

STATUS_NAMES = {
    0: "TIM_OK", 1: "TIM_ERR_INVALID_ARG", 2: "TIM_ERR_SHAPE", 3: "TIM_ERR_TOKEN_RANGE",
    4: "TIM_ERR_NONFINITE", 5: "TIM_ERR_EMPTY_SEQUENCE", 6: "TIM_ERR_BAD_MASK",
    7: "TIM_ERR_WORKSPACE", 8: "TIM_ERR_CUDA", 9: "TIM_ERR_TIMEOUT",
    10: "TIM_ERR_UNSUPPORTED_DEVICE", 11: "TIM_ERR_CAPACITY",
}
STATUS = {v: k for k, v in STATUS_NAMES.items()}

SEQ_EMPTY, SEQ_BAD_MASK, SEQ_NONFINITE, SEQ_BAD_OFFSETS, SEQ_K3_OVERFLOW = 1, 2, 4, 8, 16

# numpy mirror of struct tim_seq_stats (208 bytes)
PAIR_DTYPE = np.dtype([("mismatch_count", "<i8"), ("first_div", "<i8"), ("longest_run", "<i8"),
                       ("max_abs_diff", "<f8"), ("signed_mean", "<f8"), ("mae", "<f8")])
SEQ_STATS_DTYPE = np.dtype([("n_valid", "<i8"), ("pair", PAIR_DTYPE, (3,)),
                            ("mean_log_ratio", "<f8"), ("mean_weight_move", "<f8"),
                            ("mean_same_version", "<f8"), ("k3_mean", "<f8"), ("tis_mean", "<f8"),
                            ("tis_clipped", "<i8"), ("flags", "<i4"), ("reserved", "<i4")])
assert SEQ_STATS_DTYPE.itemsize == 208

# numpy mirror of struct tim_seq_diag (200 bytes)
SEQ_DIAG_DTYPE = np.dtype([("n_valid", "<i8"), ("abs_q50", "<f8", (3,)), ("abs_q95", "<f8", (3,)),
                           ("abs_q99", "<f8", (3,)), ("prob_mae", "<f8", (3,)),
                           ("top1_flips", "<i8", (3,)), ("log_ratio_sum", "<f8"),
                           ("k1_sum", "<f8"), ("k3_sum", "<f8"), ("seq_tis", "<f8"),
                           ("ratio_err_mean", "<f8"), ("mis_mean", "<f8"), ("mis_kept", "<i8"),
                           ("w2_mean", "<f8"), ("flags", "<i4"), ("reserved", "<i4")])
assert SEQ_DIAG_DTYPE.itemsize == 200


class TimError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        self.name = STATUS_NAMES.get(int(code), f"code {code}")
        super().__init__(f"{where}: {self.name}")


_c = ctypes
_vp, _i64, _i32, _f32, _sz = _c.c_void_p, _c.c_int64, _c.c_int32, _c.c_float, _c.c_size_t

_SIGNATURES = {
    "tim_status_string": (_c.c_char_p, [_c.c_int]),
    "tim_abi_version": (_i32, []),
    "tim_workspace_init": (_c.c_int, [_vp, _sz, _vp]),
    "tim_status_sync": (_c.c_int, [_vp, _vp]),
    "tim_logprob_workspace_size": (_sz, [_i64, _i32, _i32]),
    "tim_logprob": (_c.c_int, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32, _vp, _vp, _vp,
                               _vp, _sz, _vp]),
    "tim_rmsnorm_rows": (_c.c_int, [_vp, _vp, _i64, _i32, _i32, _f32, _vp, _sz, _vp]),
    "tim_lmhead_lse": (_c.c_int, [_vp, _vp, _i64, _i32, _i32, _f32, _vp, _sz, _vp]),
    "tim_lse_finalize": (_c.c_int, [_vp, _i64, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tim_compare_workspace_size": (_sz, [_i64, _i32]),
    "tim_compare": (_c.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i64, _f32, _vp, _vp, _vp, _sz,
                               _vp]),
    "tim_compare_diag_workspace_size": (_sz, [_i64, _i32]),
    "tim_quantize_fp8_rows": (_c.c_int, [_vp, _i64, _i32, _vp, _vp, _vp]),
    "tim_logprob_fp8_workspace_size": (_sz, [_i64, _i32, _i32]),
    "tim_logprob_fp8": (_c.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32, _vp, _vp,
                                   _vp, _vp, _sz, _vp]),
    "tim_split_tf32": (_c.c_int, [_vp, _i64, _vp, _vp, _vp]),
    "tim_logprob_fp32_workspace_size": (_sz, [_i64, _i32, _i32]),
    "tim_logprob_fp32": (_c.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32, _vp, _vp,
                                    _vp, _vp, _sz, _vp]),
    "tim_logprob_backward_workspace_size": (_sz, [_i64, _i32, _i32]),
    "tim_logprob_backward": (_c.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _f32,
                                        _f32, _vp, _vp, _i32, _vp, _sz, _vp]),
    "tim_logprob_noalloc": (_c.c_int, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32, _vp, _vp,
                                       _vp, _vp, _vp]),
    "tim_selftest_workspace_size": (_sz, []),
    "tim_selftest_wait_timeout": (_c.c_int, [_i32, _vp, _sz, _vp]),
    "tim_rmsnorm_backward_workspace_size": (_sz, [_i64, _i32]),
    "tim_rmsnorm_backward": (_c.c_int, [_vp, _vp, _vp, _i64, _i32, _f32, _vp, _vp, _i32, _vp, _sz,
                                        _vp]),
    "tim_processed_logprob_workspace_size": (_sz, [_i64, _i32, _i32]),
    "tim_processed_logprob_head": (_c.c_int, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32,
                                              _i32, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                              _vp]),
    "tim_processed_logprob": (_c.c_int, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32, _i32,
                                         _f32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tim_vocab_shard": (_c.c_int, [_i32, _i32, _i32, _c.POINTER(_i32), _c.POINTER(_i32)]),
    "tim_logprob_shard_workspace_size": (_sz, [_i64, _i32, _i32, _i32, _i32]),
    "tim_logprob_shard": (_c.c_int, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _f32, _f32,
                                     _vp, _vp, _vp, _sz, _vp]),
    "tim_logprob_merge_workspace_size": (_sz, [_i64]),
    "tim_logprob_merge_shards": (_c.c_int, [_vp, _vp, _vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp,
                                            _sz, _vp]),
    "tim_compare_diag": (_c.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i64, _f32,
                                    _f32, _f32, _vp, _vp, _sz, _vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libtim.so (built in-tree by ``build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtim.so not found at {LIB_PATH}: run __graft_entry__.build() "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().tim_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != 0:
        raise TimError(code, where)


# ----------------------------------------------------------------------------- torch helpers

def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _ptr(t) -> int:
    return t.data_ptr()


def _need(t, dtype, name, ndim=None, cuda=True):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D")


class Workspace:
    """A device workspace (torch uint8 buffer) with its status word zeroed once."""

    def __init__(self, nbytes: int, device=None, stream=None):
        torch = _torch()
        self.nbytes = int(max(nbytes, 1024))
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        if self.buf.data_ptr() % 256:
            raise RuntimeError("workspace is not 256-byte aligned")
        _check(lib().tim_workspace_init(self.ptr, self.nbytes, _stream_ptr(stream)),
               "tim_workspace_init")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def sync_status(self, stream=None) -> int:
        return int(lib().tim_status_sync(self.ptr, _stream_ptr(stream)))

    def check(self, where: str = "kernel", stream=None):
        code = self.sync_status(stream)
        if code != 0:
            raise TimError(code, where)


def logprob_workspace_size(T: int, d: int, V: int) -> int:
    return int(lib().tim_logprob_workspace_size(int(T), int(d), int(V)))


def compare_workspace_size(T: int, n_seq: int) -> int:
    return int(lib().tim_compare_workspace_size(int(T), int(n_seq)))


def _as_bf16(t, name):
    """Accept bf16 tensors or 16-bit integer views of bf16 bit patterns."""
    torch = _torch()
    if t.dtype == torch.int16 or t.dtype == getattr(torch, "uint16", torch.int16):
        t = t.view(torch.bfloat16)
    _need(t, torch.bfloat16, name)
    return t


def logprob(hidden, gamma, W, token_ids, temperature: float, eps: float, *, out=None,
            workspace: Optional[Workspace] = None, stream=None, check: bool = True):
    """Score rows with tim_logprob.  Returns (logprob f32 [T], lse f32 [T], top1 i32 [T]).

    hidden bf16 [T, d], gamma bf16 [d], W bf16 [V, d], token_ids int32 [T] (CUDA tensors;
    int16 views of bf16 bits are accepted).  ``check`` synchronises and raises on a
    data-dependent error.
    """
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    W = _as_bf16(W, "W")
    _need(token_ids, torch.int32, "token_ids", 1)
    T, d = hidden.shape
    V = W.shape[0]
    if W.shape[1] != d or gamma.shape != (d,) or token_ids.shape[0] != T:
        raise ValueError("shape mismatch between hidden, gamma, W and token_ids")
    if out is None:
        out = (torch.empty(T, dtype=torch.float32, device=hidden.device),
               torch.empty(T, dtype=torch.float32, device=hidden.device),
               torch.empty(T, dtype=torch.int32, device=hidden.device))
    lp, lse, top1 = out
    if workspace is None:
        workspace = Workspace(logprob_workspace_size(T, d, V), hidden.device, stream)
    code = lib().tim_logprob(_ptr(hidden), _ptr(gamma), _ptr(W), _ptr(token_ids), T, d, V,
                             float(temperature), float(eps), _ptr(lp), _ptr(lse), _ptr(top1),
                             workspace.ptr, workspace.nbytes, _stream_ptr(stream))
    _check(code, "tim_logprob")
    if check:
        workspace.check("tim_logprob", stream)
    return lp, lse, top1


def logprob_stages(hidden, gamma, W, token_ids, temperature: float, eps: float, out,
                   workspace: Workspace, stream=None, events=None):
    """The three stages of tim_logprob as separate C-ABI calls (same work, same order).

    ``events`` = optional list of 4 torch.cuda.Event recorded before stage 1, between the
    stages and after stage 3 on ``stream``.
    """
    T, d = hidden.shape
    V = W.shape[0]
    lp, lse, top1 = out
    sp = _stream_ptr(stream)
    L = lib()
    ev = events or [None] * 4
    if ev[0] is not None:
        ev[0].record(stream)
    _check(L.tim_rmsnorm_rows(_ptr(hidden), _ptr(gamma), T, d, V, float(eps), workspace.ptr,
                              workspace.nbytes, sp), "tim_rmsnorm_rows")
    if ev[1] is not None:
        ev[1].record(stream)
    _check(L.tim_lmhead_lse(_ptr(W), _ptr(token_ids), T, d, V, float(temperature), workspace.ptr,
                            workspace.nbytes, sp), "tim_lmhead_lse")
    if ev[2] is not None:
        ev[2].record(stream)
    _check(L.tim_lse_finalize(_ptr(token_ids), T, d, V, float(temperature), _ptr(lp), _ptr(lse),
                              _ptr(top1), workspace.ptr, workspace.nbytes, sp), "tim_lse_finalize")
    if ev[3] is not None:
        ev[3].record(stream)


def compare(lp_gen, lp_replay, lp_train, seq_offsets, mask, tis_cap: float, *, out_stats=None,
            out_tis_w=None, want_tis_w: bool = True, workspace: Optional[Workspace] = None,
            stream=None, check: bool = True, to_host: bool = True):
    """Per-sequence A/B/C statistics with tim_compare.

    lp_* float32 [T], seq_offsets int64 [S+1], mask uint8 [T] (CUDA tensors).
    Returns (stats, tis_w): stats is a numpy structured array (SEQ_STATS_DTYPE) when
    ``to_host`` else the raw device uint8 buffer.
    """
    torch = _torch()
    for t, n in ((lp_gen, "lp_gen"), (lp_replay, "lp_replay"), (lp_train, "lp_train")):
        _need(t, torch.float32, n, 1)
    _need(seq_offsets, torch.int64, "seq_offsets", 1)
    _need(mask, torch.uint8, "mask", 1)
    T = lp_gen.shape[0]
    S = seq_offsets.shape[0] - 1
    if lp_replay.shape[0] != T or lp_train.shape[0] != T or mask.shape[0] != T or S < 1:
        raise ValueError("shape mismatch")
    dev = lp_gen.device
    if out_stats is None:
        out_stats = torch.empty(S * SEQ_STATS_DTYPE.itemsize, dtype=torch.uint8, device=dev)
    if out_tis_w is None and want_tis_w:
        out_tis_w = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = Workspace(compare_workspace_size(T, S), dev, stream)
    code = lib().tim_compare(_ptr(lp_gen), _ptr(lp_replay), _ptr(lp_train), _ptr(seq_offsets), S,
                             _ptr(mask), T, float(tis_cap), _ptr(out_stats),
                             _ptr(out_tis_w) if out_tis_w is not None else None,
                             workspace.ptr, workspace.nbytes, _stream_ptr(stream))
    _check(code, "tim_compare")
    if check:
        workspace.check("tim_compare", stream)
    if to_host:
        host = out_stats.cpu().numpy().view(SEQ_STATS_DTYPE)
        return host, out_tis_w
    return out_stats, out_tis_w


def compare_diag(lp_gen, lp_replay, lp_train, seq_offsets, mask, tis_cap: float,
                 mis_lo: float, mis_hi: float, top1=(None, None, None), *, out=None,
                 workspace: Optional[Workspace] = None, stream=None, check: bool = True,
                 to_host: bool = True):
    """Extended per-sequence diagnostics with tim_compare_diag.

    top1 = (top1_gen, top1_replay, top1_train), each an int32 [T] CUDA tensor or None.
    Returns a numpy structured array (SEQ_DIAG_DTYPE) when ``to_host`` else the raw
    device buffer.
    """
    torch = _torch()
    for t, n in ((lp_gen, "lp_gen"), (lp_replay, "lp_replay"), (lp_train, "lp_train")):
        _need(t, torch.float32, n, 1)
    _need(seq_offsets, torch.int64, "seq_offsets", 1)
    _need(mask, torch.uint8, "mask", 1)
    tops = []
    for t, n in zip(top1, ("top1_gen", "top1_replay", "top1_train")):
        if t is not None:
            _need(t, torch.int32, n, 1)
        tops.append(None if t is None else _ptr(t))
    T = lp_gen.shape[0]
    S = seq_offsets.shape[0] - 1
    if lp_replay.shape[0] != T or lp_train.shape[0] != T or mask.shape[0] != T or S < 1:
        raise ValueError("shape mismatch")
    dev = lp_gen.device
    if out is None:
        out = torch.empty(S * SEQ_DIAG_DTYPE.itemsize, dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = Workspace(int(lib().tim_compare_diag_workspace_size(T, S)), dev, stream)
    code = lib().tim_compare_diag(_ptr(lp_gen), _ptr(lp_replay), _ptr(lp_train), tops[0], tops[1],
                                  tops[2], _ptr(seq_offsets), S, _ptr(mask), T, float(tis_cap),
                                  float(mis_lo), float(mis_hi), _ptr(out), workspace.ptr,
                                  workspace.nbytes, _stream_ptr(stream))
    _check(code, "tim_compare_diag")
    if check:
        workspace.check("tim_compare_diag", stream)
    if to_host:
        return out.cpu().numpy().view(SEQ_DIAG_DTYPE)
    return out


def diag_to_dicts(arr) -> list:
    """Structured diag array -> list of dicts shaped like the oracle's."""
    keys3 = ("abs_q50", "abs_q95", "abs_q99", "prob_mae")
    out = []
    for r in arr:
        dct = {k: [float(v) for v in r[k]] for k in keys3}
        dct["top1_flips"] = [int(v) for v in r["top1_flips"]]
        for k in ("log_ratio_sum", "k1_sum", "k3_sum", "seq_tis", "ratio_err_mean", "mis_mean",
                  "w2_mean"):
            dct[k] = float(r[k])
        dct["n_valid"] = int(r["n_valid"])
        dct["mis_kept"] = int(r["mis_kept"])
        dct["flags"] = int(r["flags"])
        out.append(dct)
    return out


def quantize_fp8_rows(x, *, stream=None):
    """Per-row e4m3 quantisation of a bf16 [rows, K] CUDA tensor: returns (codes uint8
    [rows, K], scales float32 [rows]) (tim_quantize_fp8_rows)."""
    torch = _torch()
    x = _as_bf16(x, "x")
    rows, K = x.shape
    codes = torch.empty(rows, K, dtype=torch.uint8, device=x.device)
    scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(lib().tim_quantize_fp8_rows(_ptr(x), rows, K, _ptr(codes), _ptr(scales),
                                       _stream_ptr(stream)), "tim_quantize_fp8_rows")
    return codes, scales


def logprob_fp8(hidden, gamma, W_codes, W_scales, token_ids, temperature: float, eps: float, *,
                out=None, workspace: Optional[Workspace] = None, stream=None, check: bool = True):
    """FP8-head score (tim_logprob_fp8) with W quantised by quantize_fp8_rows.
    Returns (logprob, lse, top1) like ``logprob``."""
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    _need(W_codes, torch.uint8, "W_codes", 2)
    _need(W_scales, torch.float32, "W_scales", 1)
    _need(token_ids, torch.int32, "token_ids", 1)
    T, d = hidden.shape
    V = W_codes.shape[0]
    dev = hidden.device
    if out is None:
        out = (torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = Workspace(int(lib().tim_logprob_fp8_workspace_size(T, d, V)), dev, stream)
    code = lib().tim_logprob_fp8(_ptr(hidden), _ptr(gamma), _ptr(W_codes), _ptr(W_scales),
                                 _ptr(token_ids), T, d, V, float(temperature), float(eps),
                                 _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), workspace.ptr,
                                 workspace.nbytes, _stream_ptr(stream))
    _check(code, "tim_logprob_fp8")
    if check:
        workspace.check("tim_logprob_fp8", stream)
    return out


def split_tf32(x, *, stream=None):
    """tf32 split of an fp32 CUDA tensor (tim_split_tf32): returns (big, small), same shape."""
    torch = _torch()
    _need(x, torch.float32, "x")
    big = torch.empty_like(x)
    small = torch.empty_like(x)
    _check(lib().tim_split_tf32(_ptr(x), x.numel(), _ptr(big), _ptr(small), _stream_ptr(stream)),
           "tim_split_tf32")
    return big, small


def logprob_fp32(hidden, gamma, W_big, W_small, token_ids, temperature: float, eps: float, *,
                 out=None, workspace: Optional[Workspace] = None, stream=None, check: bool = True):
    """FP32-head score (tim_logprob_fp32) with W split by split_tf32.  Returns (logprob, lse,
    top1) like ``logprob``."""
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    _need(W_big, torch.float32, "W_big", 2)
    _need(W_small, torch.float32, "W_small", 2)
    _need(token_ids, torch.int32, "token_ids", 1)
    if W_big.shape != W_small.shape:
        raise ValueError("W_big and W_small must have the same shape")
    T, d = hidden.shape
    V = W_big.shape[0]
    dev = hidden.device
    if out is None:
        out = (torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = Workspace(int(lib().tim_logprob_fp32_workspace_size(T, d, V)), dev, stream)
    code = lib().tim_logprob_fp32(_ptr(hidden), _ptr(gamma), _ptr(W_big), _ptr(W_small),
                                  _ptr(token_ids), T, d, V, float(temperature), float(eps),
                                  _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), workspace.ptr,
                                  workspace.nbytes, _stream_ptr(stream))
    _check(code, "tim_logprob_fp32")
    if check:
        workspace.check("tim_logprob_fp32", stream)
    return out


def logprob_backward(hidden, gamma, W, token_ids, lse, grad_logprob, temperature: float,
                     eps: float, *, chunk_rows: Optional[int] = None, out_dy=None, out_dW=None,
                     workspace: Optional[Workspace] = None, stream=None, check: bool = True):
    """Backward of the linear logprob (tim_logprob_backward): returns (dy fp32 [T, d],
    dW fp32 [V, d]) for L = sum_t grad_logprob[t] * logprob[t].  ``lse`` is the forward's
    out_lse.  With ``chunk_rows`` the rows are processed in chunks (dW accumulated across
    them in chunk order), bounding the workspace to that many rows."""
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    W = _as_bf16(W, "W")
    _need(token_ids, torch.int32, "token_ids", 1)
    _need(lse, torch.float32, "lse", 1)
    _need(grad_logprob, torch.float32, "grad_logprob", 1)
    T, d = hidden.shape
    V = W.shape[0]
    dev = hidden.device
    if out_dy is None:
        out_dy = torch.empty(T, d, dtype=torch.float32, device=dev)
    if out_dW is None:
        out_dW = torch.empty(V, d, dtype=torch.float32, device=dev)
    step = T if not chunk_rows else max(1, min(int(chunk_rows), T))
    if workspace is None:
        workspace = Workspace(int(lib().tim_logprob_backward_workspace_size(step, d, V)), dev,
                              stream)
    for r0 in range(0, T, step):
        r1 = min(T, r0 + step)
        code = lib().tim_logprob_backward(
            _ptr(hidden) + r0 * d * 2, _ptr(gamma), _ptr(W), _ptr(token_ids) + r0 * 4,
            _ptr(lse) + r0 * 4, _ptr(grad_logprob) + r0 * 4, r1 - r0, d, V, float(temperature),
            float(eps), _ptr(out_dy) + r0 * d * 4, _ptr(out_dW), 0 if r0 == 0 else 1,
            workspace.ptr, workspace.nbytes, _stream_ptr(stream))
        _check(code, "tim_logprob_backward")
    if check:
        workspace.check("tim_logprob_backward", stream)
    return out_dy, out_dW


def logprob_noalloc(hidden, gamma, W, token_ids, temperature: float, eps: float, out,
                    out_status=None, *, stream=None):
    """tim_logprob_noalloc: the scoring path with the library's static scratch instead of
    a workspace, for callers that must not allocate device memory.  ``out`` = (logprob f32
    [T], lse f32 [T], top1 i32 [T]) preallocated; ``out_status`` an optional device int32
    [1] receiving the call's first data-dependent error code.  Nothing is allocated."""
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    W = _as_bf16(W, "W")
    _need(token_ids, torch.int32, "token_ids", 1)
    T, d = hidden.shape
    V = W.shape[0]
    code = lib().tim_logprob_noalloc(_ptr(hidden), _ptr(gamma), _ptr(W), _ptr(token_ids), T, d, V,
                                     float(temperature), float(eps), _ptr(out[0]), _ptr(out[1]),
                                     _ptr(out[2]),
                                     _ptr(out_status) if out_status is not None else None,
                                     _stream_ptr(stream))
    _check(code, "tim_logprob_noalloc")
    return out


def selftest_wait_timeout(limit_ms: int = 50, *, stream=None) -> str:
    """Run the bounded-wait self-test (tim_selftest_wait_timeout) and return the status name
    that tim_status_sync reports afterwards (``TIM_ERR_TIMEOUT`` when the waits gave up as
    designed)."""
    ws = Workspace(int(lib().tim_selftest_workspace_size()), stream=stream)
    _check(lib().tim_selftest_wait_timeout(int(limit_ms), ws.ptr, ws.nbytes, _stream_ptr(stream)),
           "tim_selftest_wait_timeout")
    code = lib().tim_status_sync(ws.ptr, _stream_ptr(stream))
    return STATUS_NAMES.get(int(code), f"code {code}")


def rmsnorm_backward(hidden, gamma, dy, eps: float, *, out_dh=None, out_dgamma=None,
                     accumulate_dgamma: bool = False, workspace: Optional[Workspace] = None,
                     stream=None, check: bool = True):
    """RMSNorm backward (tim_rmsnorm_backward): returns (dh fp32 [T, d], dgamma fp32 [d])
    for the upstream gradient dy fp32 [T, d] of y = RMSNorm(hidden) * gamma."""
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    _need(dy, torch.float32, "dy", 2)
    T, d = hidden.shape
    dev = hidden.device
    if out_dh is None:
        out_dh = torch.empty(T, d, dtype=torch.float32, device=dev)
    if out_dgamma is None:
        out_dgamma = torch.empty(d, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = Workspace(int(lib().tim_rmsnorm_backward_workspace_size(T, d)), dev, stream)
    _check(lib().tim_rmsnorm_backward(_ptr(hidden), _ptr(gamma), _ptr(dy), T, d, float(eps),
                                      _ptr(out_dh), _ptr(out_dgamma), int(bool(accumulate_dgamma)),
                                      workspace.ptr, workspace.nbytes, _stream_ptr(stream)),
           "tim_rmsnorm_backward")
    if check:
        workspace.check("tim_rmsnorm_backward", stream)
    return out_dh, out_dgamma


def _linear_logprob_function():
    torch = _torch()

    class LinearLogprob(torch.autograd.Function):
        """Custom autograd around the scoring kernels: the forward values are exactly
        tim_logprob's (batch-invariant), the backward recomputes the logits
        (tim_logprob_backward) and carries the gradient through the RMSNorm
        (tim_rmsnorm_backward).  Gradients of hidden, gamma and W are returned in their
        dtypes."""

        @staticmethod
        def forward(ctx, hidden, gamma, W, token_ids, temperature, eps):
            lp, lse, _ = logprob(hidden, gamma, W, token_ids, temperature, eps)
            ctx.save_for_backward(hidden, gamma, W, token_ids, lse)
            ctx.temperature, ctx.eps = float(temperature), float(eps)
            return lp

        @staticmethod
        def backward(ctx, grad_logprob):
            hidden, gamma, W, token_ids, lse = ctx.saved_tensors
            g = grad_logprob.contiguous().float()
            dy, dW = logprob_backward(hidden, gamma, W, token_ids, lse, g, ctx.temperature,
                                      ctx.eps)
            dh, dgamma = rmsnorm_backward(hidden, gamma, dy, ctx.eps)
            return (dh.to(hidden.dtype), dgamma.to(gamma.dtype), dW.to(W.dtype), None, None,
                    None)

    return LinearLogprob


def linear_logprob(hidden, gamma, W, token_ids, temperature: float, eps: float):
    """Differentiable selected-token logprob (bf16 hidden, gamma, W as torch bfloat16
    tensors): forward = tim_logprob, backward = tim_logprob_backward +
    tim_rmsnorm_backward (the bf16 rounding of y passed straight through)."""
    global _LINEAR_LOGPROB
    if _LINEAR_LOGPROB is None:
        _LINEAR_LOGPROB = _linear_logprob_function()
    return _LINEAR_LOGPROB.apply(hidden, gamma, W, token_ids, temperature, eps)


_LINEAR_LOGPROB = None


def processed_logprob(hidden, gamma, W, token_ids, temperature: float, eps: float, top_k: int,
                      top_p: float = 1.0, *, out=None, workspace: Optional[Workspace] = None,
                      stream=None, check: bool = True, head: bool = False):
    """Top-k / top-p processed score with tim_processed_logprob.
    Returns (logprob f32 [T] (-inf if filtered out), lse_kept f32 [T], kept i32 [T]); with
    ``head`` also the top-k head (ids i32 [T, K], processed logprobs f32 [T, K],
    K = min(top_k, V)) from tim_processed_logprob_head."""
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    W = _as_bf16(W, "W")
    _need(token_ids, torch.int32, "token_ids", 1)
    T, d = hidden.shape
    V = W.shape[0]
    dev = hidden.device
    if out is None:
        out = (torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = Workspace(int(lib().tim_processed_logprob_workspace_size(T, d, V)), dev, stream)
    if head:
        K = min(int(top_k), V)
        hid_ids = torch.empty(T, K, dtype=torch.int32, device=dev)
        hid_lp = torch.empty(T, K, dtype=torch.float32, device=dev)
        code = lib().tim_processed_logprob_head(
            _ptr(hidden), _ptr(gamma), _ptr(W), _ptr(token_ids), T, d, V, float(temperature),
            float(eps), int(top_k), float(top_p), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
            _ptr(hid_ids), _ptr(hid_lp), workspace.ptr, workspace.nbytes, _stream_ptr(stream))
    else:
        code = lib().tim_processed_logprob(_ptr(hidden), _ptr(gamma), _ptr(W), _ptr(token_ids), T,
                                           d, V, float(temperature), float(eps), int(top_k),
                                           float(top_p), _ptr(out[0]), _ptr(out[1]),
                                           _ptr(out[2]), workspace.ptr, workspace.nbytes,
                                           _stream_ptr(stream))
    _check(code, "tim_processed_logprob")
    if check:
        workspace.check("tim_processed_logprob", stream)
    return (*out, hid_ids, hid_lp) if head else out


# ----------------------------------------------------------------------------- vocab-parallel

def vocab_shard(V: int, G: int, g: int):
    """(v0, v_len) of rank g's vocabulary ids when V is split over G ranks."""
    v0, n = _c.c_int32(0), _c.c_int32(0)
    _check(lib().tim_vocab_shard(int(V), int(G), int(g), _c.byref(v0), _c.byref(n)),
           "tim_vocab_shard")
    return int(v0.value), int(n.value)


def logprob_shard(hidden, gamma, W_shard, token_ids, V: int, G: int, g: int, temperature: float,
                  eps: float, *, workspace: Optional[Workspace] = None, stream=None,
                  check: bool = True):
    """Rank g's part of the vocabulary-parallel score: returns (records float32 [T, 4],
    target logits float32 [T]) for the all-gather."""
    torch = _torch()
    hidden = _as_bf16(hidden, "hidden")
    gamma = _as_bf16(gamma, "gamma")
    if W_shard is not None:
        W_shard = _as_bf16(W_shard, "W_shard")
    _need(token_ids, torch.int32, "token_ids", 1)
    T, d = hidden.shape
    dev = hidden.device
    rec = torch.empty(T, 4, dtype=torch.float32, device=dev)
    tgt = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = Workspace(int(lib().tim_logprob_shard_workspace_size(T, d, V, G, g)), dev,
                              stream)
    code = lib().tim_logprob_shard(_ptr(hidden), _ptr(gamma),
                                   None if W_shard is None else _ptr(W_shard), _ptr(token_ids), T,
                                   d, int(V), int(G), int(g), float(temperature), float(eps),
                                   _ptr(rec), _ptr(tgt), workspace.ptr, workspace.nbytes,
                                   _stream_ptr(stream))
    _check(code, "tim_logprob_shard")
    if check:
        workspace.check("tim_logprob_shard", stream)
    return rec, tgt


def logprob_merge_shards(recs, tgts, token_ids, V: int, *, out=None,
                         workspace: Optional[Workspace] = None, stream=None, check: bool = True):
    """Merge [G, T, 4] records and [G, T] target logits (rank order) into
    (logprob, lse, top1)."""
    torch = _torch()
    _need(recs, torch.float32, "recs", 3)
    _need(tgts, torch.float32, "tgts", 2)
    _need(token_ids, torch.int32, "token_ids", 1)
    G, T, _ = recs.shape
    dev = recs.device
    if out is None:
        out = (torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = Workspace(int(lib().tim_logprob_merge_workspace_size(T)), dev, stream)
    code = lib().tim_logprob_merge_shards(_ptr(recs), _ptr(tgts), _ptr(token_ids), T, int(V),
                                          int(G), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                          workspace.ptr, workspace.nbytes, _stream_ptr(stream))
    _check(code, "tim_logprob_merge_shards")
    if check:
        workspace.check("tim_logprob_merge_shards", stream)
    return out


def gather_shard_records(rec, tgt, group=None):
    """All-gather every rank's (records [T, 4], targets [T]) into [G, T, 4] and [G, T] in
    rank order (the one exchange step of the vocabulary-parallel path)."""
    import torch.distributed as dist
    G = dist.get_world_size(group)
    recs = [rec.new_empty(rec.shape) for _ in range(G)]
    tgts = [tgt.new_empty(tgt.shape) for _ in range(G)]
    dist.all_gather(recs, rec.contiguous(), group=group)
    dist.all_gather(tgts, tgt.contiguous(), group=group)
    torch = _torch()
    return torch.stack(recs), torch.stack(tgts)


def logprob_vocab_parallel(hidden, gamma, W_shard, token_ids, V: int, temperature: float,
                           eps: float, group=None):
    """Vocabulary-parallel tim_logprob across the ranks of ``group`` (one GPU per rank,
    rank g holding W rows vocab_shard(V, G, g)); returns the same bits as tim_logprob."""
    import torch.distributed as dist
    G, g = dist.get_world_size(group), dist.get_rank(group)
    rec, tgt = logprob_shard(hidden, gamma, W_shard, token_ids, V, G, g, temperature, eps)
    recs, tgts = gather_shard_records(rec, tgt, group)
    return logprob_merge_shards(recs, tgts, token_ids, V)


def logprob_vocab_parallel_emulated(hidden, gamma, W, token_ids, G: int, temperature: float,
                                    eps: float):
    """The vocabulary-parallel path with G shards run one after another on this GPU."""
    torch = _torch()
    W = _as_bf16(W, "W")
    V = W.shape[0]
    recs, tgts = [], []
    for g in range(G):
        v0, n = vocab_shard(V, G, g)
        rec, tgt = logprob_shard(hidden, gamma, W[v0:v0 + n] if n else None, token_ids, V, G, g,
                                 temperature, eps)
        recs.append(rec)
        tgts.append(tgt)
    return logprob_merge_shards(torch.stack(recs), torch.stack(tgts), token_ids, V)


def stats_to_dicts(arr) -> list:
    """Structured stats array -> list of dicts shaped like the oracle's."""
    out = []
    for r in arr:
        out.append(dict(
            n_valid=int(r["n_valid"]),
            pair=[dict(mismatch_count=int(p["mismatch_count"]), first_div=int(p["first_div"]),
                       longest_run=int(p["longest_run"]), max_abs_diff=float(p["max_abs_diff"]),
                       signed_mean=float(p["signed_mean"]), mae=float(p["mae"]))
                  for p in r["pair"]],
            mean_log_ratio=float(r["mean_log_ratio"]), mean_weight_move=float(r["mean_weight_move"]),
            mean_same_version=float(r["mean_same_version"]), k3_mean=float(r["k3_mean"]),
            tis_mean=float(r["tis_mean"]), tis_clipped=int(r["tis_clipped"]),
            flags=int(r["flags"])))
    return out
