"""Deterministic fused linear-logp for GB300 (sm_103a): Python binding of liblp.so.

Every entry point of the C ABI (include/lp.h) has a function of the same name here.
This module only marshals arguments: it checks that tensors live on the GPU with the
expected dtype and layout, allocates outputs and workspace through PyTorch, takes
the current CUDA stream and calls the library. All arithmetic runs in the library's
CUDA kernels; there is no CPU path. If liblp.so has not been built, importing the
functions works but the first call raises ImportError.

    part = VocabPartition(vocab_real=151936, vocab_padded=151936, ranges=((0, 151936),))
    out = lp_forward(X, [W], None, part, y, tau=0.7)      # out["logp"], out["lse"], out["entropy"]
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence, Tuple

import torch

from . import _build
from ._build import DEBUG_LIB as _BUILT_DEBUG_LIB
from ._build import LIB as _BUILT_LIB

# The in-tree build by default; LP_LIBRARY points the binding at another build of the
# same C ABI (for example one installed elsewhere).
LIB_PATH = os.environ.get("LP_LIBRARY", _BUILT_LIB)

LP_MAX_SHARDS = 8
LP_REPLAY_SLOTS = 64
LP_NOALLOC_SCRATCH_BYTES = 32 << 20
LP_MAX_PARTS = 64

LP_OK = 0
STATUS_NAMES = {
    0: "LP_OK",
    1: "LP_ERR_INVALID_ARG",
    2: "LP_ERR_ALIGNMENT",
    3: "LP_ERR_UNSUPPORTED_DEVICE",
    4: "LP_ERR_WORKSPACE_TOO_SMALL",
    5: "LP_ERR_TARGET_OUT_OF_RANGE",
    6: "LP_ERR_REPLAY_ID_OUT_OF_RANGE",
    7: "LP_ERR_DEVICE_TIMEOUT",
    8: "LP_ERR_CUDA",
    9: "LP_ERR_REPLAY_TOO_MANY_IDS",
    10: "LP_ERR_BOUNDS",
}

LP_OP_FORWARD = 0
LP_OP_FORWARD_FROM_LOGITS = 1
LP_OP_TOP_P_REPLAY = 2
LP_OP_BACKWARD = 3
LP_OP_TOP_P_REPLAY_DENSE_MASK = 4
LP_OP_BACKWARD_FROM_LOGITS = 5
LP_OP_FORWARD_HOST = 6

LP_DTYPE_F32 = 0
LP_DTYPE_BF16 = 1
_LP_DTYPES = {torch.float32: LP_DTYPE_F32, torch.bfloat16: LP_DTYPE_BF16}

# every symbol include/lp.h declares
EXPORTED = ("lp_workspace_size", "lp_forward", "lp_forward_noalloc", "lp_forward_host", "lp_forward_from_logits",
            "lp_top_p_replay", "lp_top_p_replay_from_logits", "lp_top_p_replay_dense_mask", "lp_backward",
            "lp_backward_ex", "lp_backward_from_logits", "lp_get_device_error", "lp_selftest_wait_timeout",
            "lp_selftest_bounds", "lp_debug_bounds_build", "lp_device_supported", "lp_status_string",
            "lp_build_id", "lp_merge_shard_stats", "lp_sum_partials", "lp_set_wait_limit")


class LPError(RuntimeError):
    """A non-OK lp_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


@dataclass(frozen=True)
class VocabPartition:
    """Tensor-parallel vocabulary partition: contiguous ascending global-id ranges
    covering [0, vocab_padded), or, with local=True, only one rank's range
    [ranges[0][0], ranges[-1][1]); ids >= vocab_real are padding."""
    vocab_real: int
    vocab_padded: int
    ranges: Tuple[Tuple[int, int], ...]
    local: bool = False

    @property
    def n_shards(self) -> int:
        return len(self.ranges)


class _ShardRange(ctypes.Structure):
    _fields_ = [("vocab_start", ctypes.c_int64), ("vocab_end", ctypes.c_int64)]


class _Partition(ctypes.Structure):
    _fields_ = [("vocab_real", ctypes.c_int64), ("vocab_padded", ctypes.c_int64),
                ("n_shards", ctypes.c_int32), ("shards", ctypes.POINTER(_ShardRange)), ("local", ctypes.c_int32)]


class _Outputs(ctypes.Structure):
    _fields_ = [("logp", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("entropy", ctypes.c_void_p), ("shard_stats", ctypes.c_void_p)]


class _BackwardOptions(ctypes.Structure):
    _fields_ = [("dx_dtype", ctypes.c_int32), ("accumulate", ctypes.c_int32), ("dw_dtype", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded liblp.so (raises ImportError if it has not been built, or if an in-tree
    build was compiled from other sources than the ones beside it)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"liblp.so is not built ({LIB_PATH}); run "
                          "`python -m lm_head_linear_tcgen05_gb300._build` or __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    L.lp_build_id.argtypes = []
    L.lp_build_id.restype = ctypes.c_char_p
    built = L.lp_build_id().decode()
    in_tree = {os.path.realpath(_BUILT_LIB): False, os.path.realpath(_BUILT_DEBUG_LIB): True}
    debug = in_tree.get(os.path.realpath(LIB_PATH))
    if debug is not None:
        want = _build.source_hash(debug_bounds=debug)
        if built != want:
            raise ImportError(f"{LIB_PATH} was built from sources {built}, but the sources here hash to {want}: "
                              "rebuild it (`python -m lm_head_linear_tcgen05_gb300._build`)")
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER
    L.lp_workspace_size.argtypes = [ctypes.c_int, i64, i64, P(_Partition)]
    L.lp_workspace_size.restype = sz
    L.lp_forward.argtypes = [vp, i64, i64, P(vp), P(vp), P(_Partition), vp, f32, P(_Outputs), vp, sz, vp]
    L.lp_forward_noalloc.argtypes = [vp, i64, i64, P(vp), P(vp), P(_Partition), vp, f32, P(_Outputs), vp]
    L.lp_forward_from_logits.argtypes = [P(vp), P(i64), i64, P(_Partition), vp, f32, P(_Outputs), vp, sz, vp]
    L.lp_top_p_replay.argtypes = [vp, i64, i64, P(vp), P(vp), P(_Partition), vp, vp, f32, P(_Outputs), vp, sz, vp]
    L.lp_top_p_replay_from_logits.argtypes = [P(vp), P(i64), i64, P(_Partition), vp, vp, f32, P(_Outputs), vp, sz,
                                              vp]
    L.lp_top_p_replay_dense_mask.argtypes = [vp, i64, i64, P(vp), P(vp), P(_Partition), P(vp), vp, f32,
                                             P(_Outputs), vp, sz, vp]
    L.lp_backward.argtypes = [vp, i64, i64, P(vp), P(vp), P(_Partition), vp, f32, vp, vp, vp, vp, vp, P(vp),
                              P(vp), vp, sz, vp]
    L.lp_backward_ex.argtypes = [vp, i64, i64, P(vp), P(vp), P(_Partition), vp, f32, vp, vp, vp, vp, vp, P(vp),
                                 P(vp), P(_BackwardOptions), vp, sz, vp]
    L.lp_backward_from_logits.argtypes = [P(vp), P(i64), i64, P(_Partition), vp, f32, vp, vp, vp, vp, P(vp),
                                          P(i64), ctypes.c_int, vp]
    L.lp_forward_host.argtypes = [vp, i64, i64, P(vp), P(vp), P(_Partition), vp, f32, P(_Outputs), vp, sz, vp]
    L.lp_merge_shard_stats.argtypes = [vp, i64, P(_Partition), vp, P(_Outputs), vp]
    L.lp_sum_partials.argtypes = [P(vp), i32, i64, vp, ctypes.c_int, vp]
    L.lp_get_device_error.argtypes = [vp]
    L.lp_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    L.lp_set_wait_limit.argtypes = [ctypes.c_uint64]
    L.lp_selftest_bounds.argtypes = [vp]
    L.lp_debug_bounds_build.argtypes = []
    L.lp_device_supported.argtypes = []
    L.lp_status_string.argtypes = [ctypes.c_int]
    L.lp_status_string.restype = ctypes.c_char_p
    for name in ("lp_forward", "lp_forward_noalloc", "lp_forward_from_logits", "lp_top_p_replay",
                 "lp_top_p_replay_from_logits", "lp_top_p_replay_dense_mask",
                 "lp_backward", "lp_backward_ex", "lp_backward_from_logits", "lp_forward_host", "lp_get_device_error",
                 "lp_selftest_wait_timeout", "lp_selftest_bounds", "lp_debug_bounds_build", "lp_device_supported",
                 "lp_merge_shard_stats", "lp_sum_partials", "lp_set_wait_limit"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def use_library(path: str) -> ctypes.CDLL:
    """Load the library at `path` (e.g. the bounds-checked liblp_debug.so) for every later
    call of this module, in place of the one loaded so far."""
    global _lib, LIB_PATH
    LIB_PATH = path
    _lib = None
    return lib()


# ------------------------------------------------------------------ marshalling

def _c_partition(part) -> Tuple[_Partition, object]:
    n = len(part.ranges)
    arr = (_ShardRange * max(n, 1))(*[_ShardRange(int(s), int(e)) for s, e in part.ranges])
    cp = _Partition(int(part.vocab_real), int(part.vocab_padded), n, ctypes.cast(arr, ctypes.POINTER(_ShardRange)),
                    1 if getattr(part, "local", False) else 0)
    return cp, arr


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _ptr_array(ts) -> ctypes.Array:
    return (ctypes.c_void_p * max(len(ts), 1))(*[_ptr(t) for t in ts])


def _check(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(dev) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _raise(st: int, where: str):
    if st != LP_OK:
        raise LPError(st, where)


def lp_status_string(status: int) -> str:
    return lib().lp_status_string(int(status)).decode()


def lp_build_id() -> str:
    """Hash of the sources and code flags the loaded library was compiled from."""
    return lib().lp_build_id().decode()


def build_info() -> dict:
    """Which library is loaded, its build id, and whether this process compiled it."""
    info = {"library": LIB_PATH, "build_id": lp_build_id()}
    for rec in _build.BUILDS.values():
        if os.path.realpath(rec["lib"]) == os.path.realpath(LIB_PATH):
            info["compiled_in_this_process"] = bool(rec["compiled"])
            info["machine"] = rec["machine"]
    return info


def lp_device_supported() -> bool:
    return bool(lib().lp_device_supported())


def lp_workspace_size(op: int, T: int, H: int, part) -> int:
    cp, _keep = _c_partition(part)
    return int(lib().lp_workspace_size(int(op), int(T), int(H), ctypes.byref(cp)))


def lp_get_device_error(stream: Optional[int] = None) -> int:
    """Synchronise the stream and return (and clear) the sticky device error code."""
    s = _stream(torch.cuda.current_device()) if stream is None else stream
    return int(lib().lp_get_device_error(s))


def lp_debug_bounds_build() -> bool:
    """True if the loaded library was built with device-side bounds checks."""
    return bool(lib().lp_debug_bounds_build())


def lp_selftest_bounds(stream: Optional[int] = None) -> None:
    """Run the bounds-check self-test (LP_ERR_BOUNDS in the device error word of a
    bounds-checked build, nothing in the regular one)."""
    s = _stream(torch.cuda.current_device()) if stream is None else stream
    _raise(lib().lp_selftest_bounds(s), "lp_selftest_bounds")


def lp_set_wait_limit(limit_ns: int) -> None:
    """Set the pipeline wait limit of later GEMM launches (ns; 0 restores the 2 s default)."""
    _raise(lib().lp_set_wait_limit(int(limit_ns)), "lp_set_wait_limit")


def lp_selftest_wait_timeout(limit_ns: int, stream: Optional[int] = None) -> None:
    """Launch the bounded-wait self-test; lp_get_device_error() then reports 7."""
    s = _stream(torch.cuda.current_device()) if stream is None else stream
    _raise(lib().lp_selftest_wait_timeout(int(limit_ns), s), "lp_selftest_wait_timeout")


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]):
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def _outputs(T: int, n_shards: int, device, entropy: bool, shard_stats: bool, out: Optional[dict] = None):
    """Output tensors: the caller's (``out``, contiguous fp32 of the right shapes) or new ones."""
    if out is None:
        o = {"logp": torch.empty(T, dtype=torch.float32, device=device),
             "lse": torch.empty(T, dtype=torch.float32, device=device),
             "entropy": torch.empty(T, dtype=torch.float32, device=device) if entropy else None,
             "shard_stats": torch.empty((n_shards, 3, T), dtype=torch.float32, device=device) if shard_stats
             else None}
    else:
        o = {k: out.get(k) for k in ("logp", "lse", "entropy", "shard_stats")}
        for k in ("logp", "lse", "entropy"):
            if o[k] is not None:
                _check(o[k], f"out[{k!r}]", torch.float32, 1)
                if o[k].shape[0] != T:
                    raise ValueError(f"out[{k!r}] must have T entries")
        if o["logp"] is None or o["lse"] is None:
            raise ValueError("out must hold logp and lse")
        if o["shard_stats"] is not None:
            _check(o["shard_stats"], "out['shard_stats']", torch.float32, 3)
            _shape(o["shard_stats"], "out['shard_stats']", (n_shards, 3, T))
    co = _Outputs(_ptr(o["logp"]), _ptr(o["lse"]), _ptr(o["entropy"]), _ptr(o["shard_stats"]))
    return o, co


def _same_device(a: torch.Tensor, b: torch.Tensor):
    if a.device != b.device:
        raise ValueError(f"tensors on different devices ({a.device}, {b.device})")


def _shape(t: Optional[torch.Tensor], name: str, shape: tuple):
    """The library sees only pointers, so every extent it will read or write is checked here."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _shard_shapes(ts, part, name: str, inner: Optional[int] = None, rows: Optional[int] = None):
    """Per shard k: [V_k] (inner and rows None), [V_k, inner] or [rows, V_k]."""
    if ts is None:
        return
    for k, ((s0, e0), t) in enumerate(zip(part.ranges, ts)):
        w = e0 - s0
        shape = (w,) if inner is None and rows is None else ((w, inner) if rows is None else (rows, w))
        _shape(t, f"{name}[{k}]", shape)


def _shard_list(ts, n: int, name: str, dtype, ndim: int, allow_none: bool):
    if ts is None:
        return [None] * n
    if len(ts) != n:
        raise ValueError(f"{name} must have one entry per shard ({n})")
    for k, t in enumerate(ts):
        if t is None:
            if not allow_none:
                raise ValueError(f"{name}[{k}] is None")
            continue
        _check(t, f"{name}[{k}]", dtype, ndim)
    return list(ts)


# ------------------------------------------------------------------ entry points

def lp_forward(X: torch.Tensor, W: Sequence[torch.Tensor], bias: Optional[Sequence[torch.Tensor]], part,
               y: torch.Tensor, tau: float, entropy: bool = True, shard_stats: bool = False,
               workspace: Optional[torch.Tensor] = None, out: Optional[dict] = None) -> dict:
    """Fused linear-logp forward. X bf16 [T,H]; W[k] bf16 [V_k,H]; bias None or per-shard
    bf16 [V_k]; y int32 [T]. Returns dict of fp32 tensors logp, lse, entropy, shard_stats
    (written into ``out`` when given)."""
    _check(X, "X", torch.bfloat16, 2)
    _check(y, "y", torch.int32, 1)
    n = len(part.ranges)
    W = _shard_list(W, n, "W", torch.bfloat16, 2, True)
    bias = _shard_list(bias, n, "bias", torch.bfloat16, 1, True) if bias is not None else None
    T, H = X.shape
    _shape(y, "y", (T,))
    _shard_shapes(W, part, "W", inner=H)
    _shard_shapes(bias, part, "bias")
    cp, _keep = _c_partition(part)
    with torch.cuda.device(X.device):
        need = lp_workspace_size(LP_OP_FORWARD, T, H, part)
        ws, wsb = _workspace(need, X.device, workspace)
        o, co = _outputs(T, n, X.device, entropy, shard_stats, out)
        st = lib().lp_forward(X.data_ptr(), T, H, _ptr_array(W), _ptr_array(bias) if bias is not None else None,
                              ctypes.byref(cp), y.data_ptr(), float(tau), ctypes.byref(co), _ptr(ws), wsb,
                              _stream(X.device))
    _raise(st, "lp_forward")
    return o


def lp_forward_noalloc(X: torch.Tensor, W: Sequence[torch.Tensor], bias: Optional[Sequence[torch.Tensor]], part,
                       y: torch.Tensor, tau: float, entropy: bool = True, shard_stats: bool = False) -> dict:
    """lp_forward without a workspace: the library uses its own fixed device scratch
    (LP_NOALLOC_SCRATCH_BYTES per GPU), for callers that cannot allocate device memory.
    Only the outputs are allocated here, as the caller's buffers."""
    _check(X, "X", torch.bfloat16, 2)
    _check(y, "y", torch.int32, 1)
    n = len(part.ranges)
    W = _shard_list(W, n, "W", torch.bfloat16, 2, True)
    bias = _shard_list(bias, n, "bias", torch.bfloat16, 1, True) if bias is not None else None
    T, H = X.shape
    _shape(y, "y", (T,))
    _shard_shapes(W, part, "W", inner=H)
    _shard_shapes(bias, part, "bias")
    cp, _keep = _c_partition(part)
    with torch.cuda.device(X.device):
        o, co = _outputs(T, n, X.device, entropy, shard_stats)
        st = lib().lp_forward_noalloc(X.data_ptr(), T, H, _ptr_array(W),
                                      _ptr_array(bias) if bias is not None else None, ctypes.byref(cp),
                                      y.data_ptr(), float(tau), ctypes.byref(co), _stream(X.device))
    _raise(st, "lp_forward_noalloc")
    return o


def _logits_ld(logits, part, T: int):
    n = len(part.ranges)
    if len(logits) != n:
        raise ValueError("logits must have one entry per shard")
    ld = (ctypes.c_int64 * max(n, 1))()
    for k, (L, (s0, e0)) in enumerate(zip(logits, part.ranges)):
        if L is None:
            continue
        if not (isinstance(L, torch.Tensor) and L.is_cuda and L.dtype == torch.bfloat16 and L.dim() == 2):
            raise TypeError(f"logits[{k}] must be a 2-D bf16 CUDA tensor")
        if L.stride(1) != 1 or tuple(L.shape) != (T, e0 - s0):
            raise ValueError(f"logits[{k}] must be [T, V_k] = [{T}, {e0 - s0}] with unit column stride")
        ld[k] = L.stride(0)
    return ld


def lp_forward_from_logits(logits: Sequence[torch.Tensor], part, y: torch.Tensor, tau: float,
                           entropy: bool = True, shard_stats: bool = False) -> dict:
    """Logits-reuse forward from unscaled bf16 logits[k] [T, V_k] (row stride = stride(0))."""
    _check(y, "y", torch.int32, 1)
    n = len(part.ranges)
    T = y.shape[0]
    ld = _logits_ld(logits, part, T)
    cp, _keep = _c_partition(part)
    with torch.cuda.device(y.device):
        o, co = _outputs(T, n, y.device, entropy, shard_stats)
        st = lib().lp_forward_from_logits(_ptr_array(logits), ld, T, ctypes.byref(cp), y.data_ptr(), float(tau),
                                          ctypes.byref(co), None, 0, _stream(y.device))
    _raise(st, "lp_forward_from_logits")
    return o


def lp_top_p_replay(X: torch.Tensor, W, bias, part, replay_ids: torch.Tensor, y: torch.Tensor, tau: float,
                    shard_stats: bool = False) -> dict:
    """Compact top-p replay: replay_ids int32 [T, 64] (-1 = unused slot)."""
    _check(X, "X", torch.bfloat16, 2)
    _check(y, "y", torch.int32, 1)
    _check(replay_ids, "replay_ids", torch.int32, 2)
    if replay_ids.shape[1] != LP_REPLAY_SLOTS or replay_ids.shape[0] != X.shape[0]:
        raise ValueError("replay_ids must be [T, 64]")
    n = len(part.ranges)
    W = _shard_list(W, n, "W", torch.bfloat16, 2, True)
    bias = _shard_list(bias, n, "bias", torch.bfloat16, 1, True) if bias is not None else None
    T, H = X.shape
    _shape(y, "y", (T,))
    _shard_shapes(W, part, "W", inner=H)
    _shard_shapes(bias, part, "bias")
    cp, _keep = _c_partition(part)
    with torch.cuda.device(X.device):
        o, co = _outputs(T, n, X.device, False, shard_stats)
        st = lib().lp_top_p_replay(X.data_ptr(), T, H, _ptr_array(W), _ptr_array(bias) if bias is not None else None,
                                   ctypes.byref(cp), replay_ids.data_ptr(), y.data_ptr(), float(tau),
                                   ctypes.byref(co), None, 0, _stream(X.device))
    _raise(st, "lp_top_p_replay")
    return o


def lp_top_p_replay_from_logits(logits: Sequence[torch.Tensor], part, replay_ids: torch.Tensor, y: torch.Tensor,
                                tau: float, shard_stats: bool = False) -> dict:
    """Compact top-p replay scored from reused unscaled bf16 logits[k] [T, V_k]."""
    _check(y, "y", torch.int32, 1)
    _check(replay_ids, "replay_ids", torch.int32, 2)
    T = y.shape[0]
    if replay_ids.shape != (T, LP_REPLAY_SLOTS):
        raise ValueError("replay_ids must be [T, 64]")
    n = len(part.ranges)
    ld = _logits_ld(logits, part, T)
    cp, _keep = _c_partition(part)
    with torch.cuda.device(y.device):
        o, co = _outputs(T, n, y.device, False, shard_stats)
        st = lib().lp_top_p_replay_from_logits(_ptr_array(logits), ld, T, ctypes.byref(cp), replay_ids.data_ptr(),
                                               y.data_ptr(), float(tau), ctypes.byref(co), None, 0,
                                               _stream(y.device))
    _raise(st, "lp_top_p_replay_from_logits")
    return o


def lp_top_p_replay_dense_mask(X: torch.Tensor, W, bias, part, keep_mask: Sequence[torch.Tensor], y: torch.Tensor,
                               tau: float, shard_stats: bool = False,
                               workspace: Optional[torch.Tensor] = None) -> dict:
    """Dense keep-mask route: keep_mask[k] uint8 [T, V_k]; bitwise equal to lp_top_p_replay."""
    _check(X, "X", torch.bfloat16, 2)
    _check(y, "y", torch.int32, 1)
    n = len(part.ranges)
    W = _shard_list(W, n, "W", torch.bfloat16, 2, True)
    bias = _shard_list(bias, n, "bias", torch.bfloat16, 1, True) if bias is not None else None
    keep_mask = _shard_list(keep_mask, n, "keep_mask", torch.uint8, 2, True)
    T, H = X.shape
    _shape(y, "y", (T,))
    _shard_shapes(W, part, "W", inner=H)
    _shard_shapes(bias, part, "bias")
    _shard_shapes(keep_mask, part, "keep_mask", rows=T)
    cp, _keep = _c_partition(part)
    with torch.cuda.device(X.device):
        need = lp_workspace_size(LP_OP_TOP_P_REPLAY_DENSE_MASK, T, H, part)
        ws, wsb = _workspace(need, X.device, workspace)
        o, co = _outputs(T, n, X.device, False, shard_stats)
        st = lib().lp_top_p_replay_dense_mask(X.data_ptr(), T, H, _ptr_array(W),
                                              _ptr_array(bias) if bias is not None else None, ctypes.byref(cp),
                                              _ptr_array(keep_mask), y.data_ptr(), float(tau), ctypes.byref(co),
                                              _ptr(ws), wsb, _stream(X.device))
    _raise(st, "lp_top_p_replay_dense_mask")
    return o


def _backward(fn: str, X: torch.Tensor, W, bias, part, y, tau, lse, grad_logp, bias_grad, workspace, entropy,
              grad_entropy, dx_dtype, accumulate, dW, db, dw_dtype=torch.float32) -> dict:
    _check(X, "X", torch.bfloat16, 2)
    _check(y, "y", torch.int32, 1)
    _check(lse, "lse", torch.float32, 1)
    _check(grad_logp, "grad_logp", torch.float32, 1)
    if (entropy is None) != (grad_entropy is None):
        raise ValueError("entropy and grad_entropy go together")
    if entropy is not None:
        _check(entropy, "entropy", torch.float32, 1)
        _check(grad_entropy, "grad_entropy", torch.float32, 1)
    if dx_dtype not in _LP_DTYPES or dw_dtype not in _LP_DTYPES:
        raise TypeError("dx_dtype and dw_dtype must be torch.float32 or torch.bfloat16")
    if accumulate and dw_dtype != torch.float32:
        raise ValueError("accumulation needs fp32 dW")
    n = len(part.ranges)
    W = _shard_list(W, n, "W", torch.bfloat16, 2, True)
    bias = _shard_list(bias, n, "bias", torch.bfloat16, 1, True) if bias is not None else None
    T, H = X.shape
    for t, nm in ((y, "y"), (lse, "lse"), (grad_logp, "grad_logp"), (entropy, "entropy"),
                  (grad_entropy, "grad_entropy")):
        _shape(t, nm, (T,))
    _shard_shapes(W, part, "W", inner=H)
    _shard_shapes(bias, part, "bias")
    widths = [e - s for s, e in part.ranges]
    if accumulate and (dW is None or (bias_grad and db is None)):
        raise ValueError("accumulate=True adds into the caller's dW (and db): pass them")
    if dW is not None:
        dW = _shard_list(dW, n, "dW", dw_dtype, 2, True)
        for k, (t, w) in enumerate(zip(dW, widths)):
            if w and (t is None or tuple(t.shape) != (w, H)):
                raise ValueError(f"dW[{k}] must be {dw_dtype} [{w}, {H}]")
    if db is not None:
        db = _shard_list(db, n, "db", torch.float32, 1, True)
        for k, (t, w) in enumerate(zip(db, widths)):
            if w and (t is None or t.shape[0] != w):
                raise ValueError(f"db[{k}] must be fp32 [{w}]")
    cp, _keep = _c_partition(part)
    with torch.cuda.device(X.device):
        need = lp_workspace_size(LP_OP_BACKWARD, T, H, part)
        ws, wsb = _workspace(need, X.device, workspace)
        dX = torch.empty((T, H), dtype=dx_dtype, device=X.device)
        if dW is None:
            dW = [torch.empty((w, H), dtype=dw_dtype, device=X.device) if w else None for w in widths]
        if db is None and bias_grad:
            db = [torch.empty(w, dtype=torch.float32, device=X.device) if w else None for w in widths]
        if not bias_grad:
            db = None
        args = [X.data_ptr(), T, H, _ptr_array(W), _ptr_array(bias) if bias is not None else None,
                ctypes.byref(cp), y.data_ptr(), float(tau), lse.data_ptr(), grad_logp.data_ptr(),
                _ptr(entropy), _ptr(grad_entropy), dX.data_ptr(), _ptr_array(dW),
                _ptr_array(db) if db is not None else None]
        if fn == "lp_backward_ex":
            opts = _BackwardOptions(_LP_DTYPES[dx_dtype], 1 if accumulate else 0, _LP_DTYPES[dw_dtype])
            args.append(ctypes.byref(opts))
        st = getattr(lib(), fn)(*args, _ptr(ws), wsb, _stream(X.device))
    _raise(st, fn)
    return {"dX": dX, "dW": dW, "db": db}


def lp_backward(X: torch.Tensor, W, bias, part, y: torch.Tensor, tau: float, lse: torch.Tensor,
                grad_logp: torch.Tensor, bias_grad: bool = True,
                workspace: Optional[torch.Tensor] = None, entropy: Optional[torch.Tensor] = None,
                grad_entropy: Optional[torch.Tensor] = None) -> dict:
    """Backward of sum_t grad_logp[t] logp[t] (+ sum_t grad_entropy[t] entropy[t]): returns
    fp32 dX [T,H], dW (per shard [V_k,H]), db (per shard [V_k], or None). `lse` and
    `entropy` are the merged outputs of lp_forward."""
    return _backward("lp_backward", X, W, bias, part, y, tau, lse, grad_logp, bias_grad, workspace, entropy,
                     grad_entropy, torch.float32, False, None, None)


def lp_backward_ex(X: torch.Tensor, W, bias, part, y: torch.Tensor, tau: float, lse: torch.Tensor,
                   grad_logp: torch.Tensor, bias_grad: bool = True, workspace: Optional[torch.Tensor] = None,
                   entropy: Optional[torch.Tensor] = None, grad_entropy: Optional[torch.Tensor] = None,
                   dx_dtype=torch.float32, accumulate: bool = False, dW=None, db=None,
                   dw_dtype=torch.float32) -> dict:
    """lp_backward with output options: ``dx_dtype`` / ``dw_dtype`` torch.float32 or
    torch.bfloat16 (the fp32 result rounded once); ``accumulate`` adds the weight and bias
    gradients into the caller's fp32 ``dW`` / ``db`` lists (otherwise those, when given,
    are overwritten)."""
    return _backward("lp_backward_ex", X, W, bias, part, y, tau, lse, grad_logp, bias_grad, workspace, entropy,
                     grad_entropy, dx_dtype, accumulate, dW, db, dw_dtype)


def lp_backward_from_logits(logits: Sequence[torch.Tensor], part, y: torch.Tensor, tau: float, lse: torch.Tensor,
                            grad_logp: torch.Tensor, entropy: Optional[torch.Tensor] = None,
                            grad_entropy: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                            out: Optional[Sequence[torch.Tensor]] = None) -> list:
    """Gradient with respect to the reused unscaled logits of lp_forward_from_logits: one
    [T, V_k] tensor per shard (None for an empty shard) of ``out_dtype``. ``out`` (optional)
    gives the destination tensors; ``out=logits`` (bf16) overwrites the logits in place."""
    _check(y, "y", torch.int32, 1)
    _check(lse, "lse", torch.float32, 1)
    _check(grad_logp, "grad_logp", torch.float32, 1)
    if (entropy is None) != (grad_entropy is None):
        raise ValueError("entropy and grad_entropy go together")
    if entropy is not None:
        _check(entropy, "entropy", torch.float32, 1)
        _check(grad_entropy, "grad_entropy", torch.float32, 1)
    if out_dtype not in _LP_DTYPES:
        raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
    n = len(part.ranges)
    T = y.shape[0]
    for t, nm in ((lse, "lse"), (grad_logp, "grad_logp"), (entropy, "entropy"), (grad_entropy, "grad_entropy")):
        _shape(t, nm, (T,))
    ld = _logits_ld(logits, part, T)
    widths = [e - s for s, e in part.ranges]
    if out is None:
        # rows padded to a 16-byte multiple (the row rule), handed back as [T, V_k] views
        per16 = 16 // torch.tensor([], dtype=out_dtype).element_size()
        out = [torch.empty((T, (w + per16 - 1) // per16 * per16), dtype=out_dtype, device=y.device)[:, :w]
               if w else None for w in widths]
    elif len(out) != n:
        raise ValueError("out must have one entry per shard")
    ld_out = (ctypes.c_int64 * max(n, 1))()
    for k, (t, w) in enumerate(zip(out, widths)):
        if t is None:
            continue
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == out_dtype and t.dim() == 2):
            raise TypeError(f"out[{k}] must be a 2-D {out_dtype} CUDA tensor")
        if t.stride(1) != 1 or tuple(t.shape) != (T, w):
            raise ValueError(f"out[{k}] must be [T, V_k] with unit column stride")
        ld_out[k] = t.stride(0)
    cp, _keep = _c_partition(part)
    with torch.cuda.device(y.device):
        st = lib().lp_backward_from_logits(_ptr_array(logits), ld, T, ctypes.byref(cp), y.data_ptr(), float(tau),
                                           lse.data_ptr(), grad_logp.data_ptr(), _ptr(entropy), _ptr(grad_entropy),
                                           _ptr_array(out), ld_out, _LP_DTYPES[out_dtype], _stream(y.device))
    _raise(st, "lp_backward_from_logits")
    return list(out)


def lp_forward_host(hX: torch.Tensor, W: Sequence[torch.Tensor], bias, part, hy: torch.Tensor, tau: float,
                    entropy: bool = True, shard_stats: bool = False, workspace: Optional[torch.Tensor] = None,
                    out: Optional[dict] = None, device=None) -> dict:
    """lp_forward from host memory, through the C entry point of the same name: CPU hX bf16
    [T,H] and hy int32 [T] in (page-locked for asynchronous copies), CPU fp32 logp / lse /
    entropy / shard_stats out (``out`` holds reusable page-locked tensors, else new ones are
    allocated). W and bias are CUDA tensors on ``device``. Synchronises the stream before
    returning, so the host tensors hold the results."""
    if hX.is_cuda or hy.is_cuda:
        raise ValueError("hX and hy must be host tensors")
    if hX.dtype != torch.bfloat16 or hy.dtype != torch.int32 or hX.dim() != 2 or hy.dim() != 1:
        raise TypeError("hX must be bf16 [T, H] and hy int32 [T]")
    if not (hX.is_contiguous() and hy.is_contiguous()):
        raise ValueError("hX and hy must be contiguous")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    T, H = hX.shape
    _shape(hy, "hy", (T,))
    n = len(part.ranges)
    W = _shard_list(W, n, "W", torch.bfloat16, 2, True)
    bias = _shard_list(bias, n, "bias", torch.bfloat16, 1, True) if bias is not None else None
    _shard_shapes(W, part, "W", inner=H)
    _shard_shapes(bias, part, "bias")
    pin = torch.cuda.is_available()
    if out is None:
        out = {"logp": torch.empty(T, dtype=torch.float32, pin_memory=pin),
               "lse": torch.empty(T, dtype=torch.float32, pin_memory=pin),
               "entropy": torch.empty(T, dtype=torch.float32, pin_memory=pin) if entropy else None,
               "shard_stats": torch.empty((n, 3, T), dtype=torch.float32, pin_memory=pin) if shard_stats else None}
    for k, shape in (("logp", (T,)), ("lse", (T,)), ("entropy", (T,)), ("shard_stats", (n, 3, T))):
        t = out.get(k)
        if t is None:
            if k in ("logp", "lse"):
                raise ValueError("out must hold logp and lse")
            continue
        if t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"out[{k!r}] must be a contiguous fp32 host tensor")
        _shape(t, f"out[{k!r}]", shape)
    co = _Outputs(_ptr(out["logp"]), _ptr(out["lse"]), _ptr(out.get("entropy")), _ptr(out.get("shard_stats")))
    cp, _keep = _c_partition(part)
    with torch.cuda.device(dev):
        need = lp_workspace_size(LP_OP_FORWARD_HOST, T, H, part)
        ws, wsb = _workspace(need, dev, workspace)
        stream = torch.cuda.current_stream(dev)
        st = lib().lp_forward_host(hX.data_ptr(), T, H, _ptr_array(W), _ptr_array(bias) if bias is not None else None,
                                   ctypes.byref(cp), hy.data_ptr(), float(tau), ctypes.byref(co), _ptr(ws), wsb,
                                   stream.cuda_stream)
        _raise(st, "lp_forward_host")
        stream.synchronize()
    return {k: out.get(k) for k in ("logp", "lse", "entropy", "shard_stats")}


def lp_merge_shard_stats(shard_stats: torch.Tensor, y: torch.Tensor, part, entropy: bool = True,
                         out: Optional[dict] = None) -> dict:
    """Rank-ordered reduction of per-shard statistics: shard_stats fp32 [n_shards, 3, T]
    (the shards of ``part`` in ascending order, e.g. gathered from the ranks of a
    vocabulary-parallel group), y int32 [T]. Returns fp32 logp, lse and entropy [T]."""
    _check(shard_stats, "shard_stats", torch.float32, 3)
    _check(y, "y", torch.int32, 1)
    n = len(part.ranges)
    T = y.shape[0]
    _shape(shard_stats, "shard_stats", (n, 3, T))
    _same_device(shard_stats, y)
    cp, _keep = _c_partition(part)
    with torch.cuda.device(y.device):
        o, co = _outputs(T, n, y.device, entropy, False, out)
        if o["shard_stats"] is not None:
            raise ValueError("out must not hold shard_stats")
        st = lib().lp_merge_shard_stats(shard_stats.data_ptr(), T, ctypes.byref(cp), y.data_ptr(), ctypes.byref(co),
                                        _stream(y.device))
    _raise(st, "lp_merge_shard_stats")
    return o


def lp_sum_partials(parts: Sequence[torch.Tensor], out_dtype=torch.float32,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """((parts[0] + parts[1]) + parts[2]) + ... elementwise, in exactly that order: the
    rank-ordered sum of per-rank partial results (fp32 tensors of one shape). The sum is
    returned as fp32, or rounded once to bf16."""
    if len(parts) < 1 or len(parts) > LP_MAX_PARTS:
        raise ValueError(f"between 1 and {LP_MAX_PARTS} parts")
    shape = tuple(parts[0].shape)
    for i, t in enumerate(parts):
        _check(t, f"parts[{i}]", torch.float32, len(shape))
        _shape(t, f"parts[{i}]", shape)
        _same_device(parts[0], t)
    if out_dtype not in _LP_DTYPES:
        raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty(shape, dtype=out_dtype, device=parts[0].device)
    _check(out, "out", out_dtype, len(shape))
    _shape(out, "out", shape)
    with torch.cuda.device(parts[0].device):
        st = lib().lp_sum_partials(_ptr_array(list(parts)), len(parts), parts[0].numel(), out.data_ptr(),
                                   _LP_DTYPES[out_dtype], _stream(parts[0].device))
    _raise(st, "lp_sum_partials")
    return out
