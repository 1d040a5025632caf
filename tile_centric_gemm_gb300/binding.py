"""Thin ctypes binding over libtilelink.so with the C ABI's names.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Importing this module loads the library and fails loudly when it is
missing (build it with ``python -m tile_centric_gemm_gb300.build``); there is
no fallback.  Tensors are torch tensors on the device the call runs on; the
stream is torch's current stream unless one is given.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libtilelink.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libtilelink.so not built: {_LIB_PATH} (run python -m tile_centric_gemm_gb300.build)")

lib = ctypes.CDLL(_LIB_PATH)

TL_OK, TL_ERR_INVALID, TL_ERR_CUDA, TL_ERR_TIMEOUT, TL_ERR_UNSUPPORTED, TL_ERR_INTERNAL = range(6)
TL_MODE_PULL, TL_MODE_PUSH = 0, 1
TL_SWIZZLE_ARRIVAL, TL_SWIZZLE_ROWS = 0, 1
TL_RS_BF16_PARTIALS, TL_RS_RING_ORDER = 1, 2
TL_LL_FLAG_IN_DATA, TL_LL_SEPARATE_FLAG = 0, 1
STATUS_NAMES = {0: "TL_OK", 1: "TL_ERR_INVALID", 2: "TL_ERR_CUDA", 3: "TL_ERR_TIMEOUT",
                4: "TL_ERR_UNSUPPORTED", 5: "TL_ERR_INTERNAL"}

# Every symbol the header declares; tests check that the library exports all of them.
EXPORTED = [
    "tl_version", "tl_last_error", "tl_signals_create", "tl_signals_destroy", "tl_signals_flags",
    "tl_signals_reset", "tl_tile_notify", "tl_tile_wait", "tl_query_status",
    "tl_gemm_workspace_size", "tl_gemm", "tl_ag_gemm_workspace_size", "tl_ag_gemm_num_flags",
    "tl_ag_gemm_tile_order", "tl_ag_gemm",
    "tl_gemm_rs_workspace_size", "tl_gemm_rs_num_flags", "tl_gemm_rs", "tl_gemm_rs_noalloc",
    "tl_moe_workspace_size", "tl_moe_num_flags", "tl_moe_ag_gemm", "tl_allgather", "tl_reduce_scatter",
    "tl_moe_down_workspace_size", "tl_moe_down_num_flags", "tl_moe_down",
    "tl_ag_attn_num_flags", "tl_ag_attn", "tl_allgather_ll_link_bytes", "tl_allgather_ll",
    "tl_test_hold_chunks",
]


class TLError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_vp = ctypes.c_void_p


class tl_ag_gemm_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("self_rank", ctypes.c_int32), ("M_shard", ctypes.c_int32),
        ("K", ctypes.c_int32), ("N", ctypes.c_int32), ("mode", ctypes.c_int32),
        ("rows_per_barrier", ctypes.c_int32), ("swizzle", ctypes.c_int32),
        ("A_shards", ctypes.POINTER(_vp)), ("B", _vp), ("gathered", _vp), ("C", _vp), ("C_f32", _vp),
        ("signals", _vp), ("src_ready", _vp),
        ("epoch", ctypes.c_uint32), ("reserved1", ctypes.c_uint32),
        ("timeout_ns", ctypes.c_uint64), ("trace", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
    ]


class tl_ag_attn_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("self_rank", ctypes.c_int32), ("S_shard", ctypes.c_int32),
        ("H", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("causal", ctypes.c_int32), ("scale", ctypes.c_float),
        ("Q", _vp), ("K_shards", ctypes.POINTER(_vp)), ("V_shards", ctypes.POINTER(_vp)),
        ("K_gathered", _vp), ("V_gathered", _vp), ("O", _vp), ("lse", _vp), ("signals", _vp),
        ("epoch", ctypes.c_uint32), ("reserved0", ctypes.c_uint32), ("timeout_ns", ctypes.c_uint64),
    ]


class tl_gemm_args(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("A", _vp), ("B", _vp), ("C", _vp), ("C_f32", _vp), ("signals", _vp), ("timeout_ns", ctypes.c_uint64),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
    ]


class tl_gemm_rs_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("M", ctypes.c_int32), ("K_r", ctypes.c_int32), ("N", ctypes.c_int32),
        ("A", ctypes.POINTER(_vp)), ("B", ctypes.POINTER(_vp)), ("out", ctypes.POINTER(_vp)),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("signals", _vp),
        ("epoch", ctypes.c_uint32), ("options", ctypes.c_uint32), ("timeout_ns", ctypes.c_uint64),
        ("trace", _vp),
    ]


class tl_moe_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("self_rank", ctypes.c_int32), ("T_r", ctypes.c_int32), ("H", ctypes.c_int32),
        ("N", ctypes.c_int32), ("E", ctypes.c_int32), ("topk", ctypes.c_int32), ("rows_per_barrier", ctypes.c_int32),
        ("X", ctypes.POINTER(_vp)), ("topk_ids", _vp), ("W", ctypes.POINTER(_vp)), ("sorted_tokens", _vp),
        ("Y", _vp), ("perm", _vp), ("expert_offsets", _vp), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("signals", _vp), ("epoch", ctypes.c_uint32), ("mode", ctypes.c_int32),
        ("timeout_ns", ctypes.c_uint64), ("trace", _vp),
    ]


class tl_moe_down_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("T_r", ctypes.c_int32), ("topk", ctypes.c_int32), ("E", ctypes.c_int32),
        ("I_r", ctypes.c_int32), ("Hd", ctypes.c_int32),
        ("H", ctypes.POINTER(_vp)), ("W2", ctypes.POINTER(_vp)), ("gates", _vp), ("routing", _vp),
        ("out", ctypes.POINTER(_vp)), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("signals", _vp),
        ("epoch", ctypes.c_uint32), ("options", ctypes.c_uint32), ("timeout_ns", ctypes.c_uint64),
    ]


class tl_allgather_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("self_rank", ctypes.c_int32), ("M_shard", ctypes.c_int32), ("K", ctypes.c_int32),
        ("mode", ctypes.c_int32), ("rows_per_barrier", ctypes.c_int32), ("A_shards", ctypes.POINTER(_vp)),
        ("gathered", _vp), ("signals", _vp), ("src_ready", _vp), ("epoch", ctypes.c_uint32),
        ("reserved0", ctypes.c_uint32), ("timeout_ns", ctypes.c_uint64),
    ]


class tl_allgather_ll_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("self_rank", ctypes.c_int32), ("M_shard", ctypes.c_int32), ("K", ctypes.c_int32),
        ("protocol", ctypes.c_int32), ("rows_per_barrier", ctypes.c_int32), ("A_shards", ctypes.POINTER(_vp)),
        ("link", _vp), ("link_bytes", ctypes.c_size_t), ("gathered", _vp), ("signals", _vp),
        ("send_mask", ctypes.c_uint64), ("epoch", ctypes.c_uint32), ("reserved0", ctypes.c_uint32),
        ("timeout_ns", ctypes.c_uint64),
    ]


class tl_reduce_scatter_args(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("M", ctypes.c_int32), ("N", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("partials", ctypes.POINTER(_vp)), ("out", ctypes.POINTER(_vp)),
    ]


def _decl(name, restype, *argtypes):
    f = getattr(lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_i, _u32, _u64, _sz = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t
_decl("tl_version", _i)
_decl("tl_last_error", ctypes.c_char_p)
_decl("tl_signals_create", _i, _i, ctypes.POINTER(_vp))
_decl("tl_signals_destroy", _i, _vp)
_decl("tl_signals_flags", _i, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_i))
_decl("tl_signals_reset", _i, _vp, _vp)
_decl("tl_tile_notify", _i, _vp, _i, _i, _u32, _vp)
_decl("tl_tile_wait", _i, _vp, _i, _i, _u32, _u64, _vp)
_decl("tl_query_status", _i, _vp, _vp, ctypes.POINTER(_i), ctypes.POINTER(_i))
_decl("tl_gemm_workspace_size", _sz, _i, _i, _i, _i)
_decl("tl_gemm", _i, ctypes.POINTER(tl_gemm_args), _vp)
_decl("tl_ag_gemm_workspace_size", _sz, _i, _i, _i, _i, _i)
_decl("tl_ag_gemm_num_flags", _i, _i, _i, _i, _i, ctypes.POINTER(_i))
_decl("tl_ag_gemm_tile_order", _i, _i, _i, _i, ctypes.POINTER(ctypes.c_int32), _i)
_decl("tl_ag_gemm", _i, ctypes.POINTER(tl_ag_gemm_args), _vp)
_decl("tl_gemm_rs_workspace_size", _sz, _i, _i, _i)
_decl("tl_moe_down_workspace_size", _sz, _i, _i, _i, _i, _i)
_decl("tl_moe_down_num_flags", _i, _i, _i, _i, _i, _i)
_decl("tl_moe_down", _i, ctypes.POINTER(tl_moe_down_args), _vp)
_decl("tl_gemm_rs_num_flags", _i, _i, _i, _i)
_decl("tl_gemm_rs", _i, ctypes.POINTER(tl_gemm_rs_args), _vp)
_decl("tl_gemm_rs_noalloc", _i, ctypes.POINTER(tl_gemm_rs_args), _vp, _vp)
_decl("tl_moe_workspace_size", _sz, _i, _i, _i, _i)
_decl("tl_moe_num_flags", _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_i))
_decl("tl_moe_ag_gemm", _i, ctypes.POINTER(tl_moe_args), _vp)
_decl("tl_allgather", _i, ctypes.POINTER(tl_allgather_args), _vp)
_decl("tl_reduce_scatter", _i, ctypes.POINTER(tl_reduce_scatter_args), _vp)
_decl("tl_allgather_ll_link_bytes", _sz, _i, _i, _i, _i)
_decl("tl_allgather_ll", _i, ctypes.POINTER(tl_allgather_ll_args), _vp)
_decl("tl_test_hold_chunks", _i, _i, _i, _u64)
_decl("tl_ag_attn_num_flags", _i, _i, _i)
_decl("tl_ag_attn", _i, ctypes.POINTER(tl_ag_attn_args), _vp)


def _check(code):
    if code != TL_OK:
        raise TLError(code, lib.tl_last_error().decode(errors="replace"))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _ptr_array(ts):
    arr = (_vp * len(ts))(*[t.data_ptr() for t in ts])
    return arr


def tl_version():
    return lib.tl_version()


def tl_last_error():
    return lib.tl_last_error().decode(errors="replace")


class Signals:
    """Owner of a tl_signals object (device flags + status word)."""

    def __init__(self, num_flags: int):
        h = _vp()
        _check(lib.tl_signals_create(int(num_flags), ctypes.byref(h)))
        self.handle = h
        self.num_flags = int(num_flags)

    def flags_ptr(self):
        p, n = _vp(), _i()
        _check(lib.tl_signals_flags(self.handle, ctypes.byref(p), ctypes.byref(n)))
        return p.value, n.value

    def flags_tensor(self):
        """A zero-copy torch uint32-as-int32 CUDA view of the flags (memory owned by the library)."""
        ptr, n = self.flags_ptr()
        return _device_view(ptr, n, "<i4")

    def read_flags(self):
        """The flags as a CPU numpy uint32 array (synchronises the device)."""
        import numpy as np
        import torch
        torch.cuda.synchronize()
        return self.flags_tensor().cpu().numpy().view(np.uint32)

    def close(self):
        if self.handle:
            lib.tl_signals_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _device_view(dev_ptr, n, typestr):
    """A torch CUDA tensor viewing n elements at dev_ptr (no copy)."""
    import torch

    class _CAI:
        def __init__(self):
            self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (dev_ptr, False),
                                             "version": 3, "strides": None}
    return torch.as_tensor(_CAI(), device="cuda")


def tl_signals_reset(sig: Signals, stream=None):
    _check(lib.tl_signals_reset(sig.handle, _stream(stream)))


def tl_tile_notify(sig: Signals, first: int, count: int, value: int, stream=None):
    _check(lib.tl_tile_notify(sig.handle, int(first), int(count), int(value) & 0xFFFFFFFF, _stream(stream)))


def tl_tile_wait(sig: Signals, first: int, count: int, value: int, timeout_ns: int = 0, stream=None):
    _check(lib.tl_tile_wait(sig.handle, int(first), int(count), int(value) & 0xFFFFFFFF, int(timeout_ns),
                            _stream(stream)))


def tl_query_status(sig: Signals, stream=None):
    """Returns (code, where); code 0 = no device error.  Clears the status word."""
    code, where = _i(), _i()
    rc = lib.tl_query_status(sig.handle, _stream(stream), ctypes.byref(code), ctypes.byref(where))
    if rc not in (TL_OK,) and code.value == 0:
        _check(rc)
    return code.value, where.value


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def tl_gemm_workspace_size(M, N, K, sm_count=0):
    return int(lib.tl_gemm_workspace_size(M, N, K, sm_count))


def tl_ag_gemm_workspace_size(R, M_shard, K, N, sm_count=0):
    return int(lib.tl_ag_gemm_workspace_size(R, M_shard, K, N, sm_count))


def tl_gemm(A, B, C, signals: Signals, *, C_f32=None, timeout_ns=0, workspace=None, stream=None):
    """C = A . B (bf16 in, fp32 accumulate) with no communication; split over K
    when the tiles leave SMs idle and a (zeroed) workspace is given."""
    M, K = A.shape
    N = B.shape[1]
    a = tl_gemm_args(M=M, N=N, K=K, reserved0=0, A=_ptr(A), B=_ptr(B), C=_ptr(C), C_f32=_ptr(C_f32),
                     signals=signals.handle, timeout_ns=int(timeout_ns), workspace=_ptr(workspace),
                     workspace_bytes=_nbytes(workspace))
    _check(lib.tl_gemm(ctypes.byref(a), _stream(stream)))


def tl_ag_gemm_num_flags(R, M_shard, K, rows_per_barrier=0):
    eff = _i()
    n = lib.tl_ag_gemm_num_flags(R, M_shard, K, rows_per_barrier, ctypes.byref(eff))
    return n, eff.value


def tl_ag_gemm_tile_order(R, self_rank, M_shard):
    Mt = -(-R * M_shard // 256)
    out = (ctypes.c_int32 * Mt)()
    _check(lib.tl_ag_gemm_tile_order(R, self_rank, M_shard, out, Mt))
    return list(out)


def tl_ag_gemm(A_shards, B, gathered, C, signals: Signals, epoch: int, *, self_rank=0, C_f32=None,
               mode=TL_MODE_PUSH, src_ready: Signals | None = None, rows_per_barrier=0, timeout_ns=0,
               trace=None, swizzle=TL_SWIZZLE_ARRIVAL, workspace=None, stream=None):
    """C = [A_0; ...; A_{R-1}] . B, gathered rows written to `gathered` (see tilelink.h)."""
    R = len(A_shards)
    M_shard, K = A_shards[0].shape
    N = B.shape[1]
    ptrs = _ptr_array(A_shards)
    a = tl_ag_gemm_args(R=R, self_rank=self_rank, M_shard=M_shard, K=K, N=N, mode=mode,
                        rows_per_barrier=rows_per_barrier, swizzle=int(swizzle),
                        A_shards=ctypes.cast(ptrs, ctypes.POINTER(_vp)), B=_ptr(B), gathered=_ptr(gathered),
                        C=_ptr(C), C_f32=_ptr(C_f32), signals=signals.handle,
                        src_ready=src_ready.handle if src_ready is not None else None,
                        epoch=int(epoch) & 0xFFFFFFFF, reserved1=0, timeout_ns=int(timeout_ns), trace=_ptr(trace),
                        workspace=_ptr(workspace), workspace_bytes=_nbytes(workspace))
    _check(lib.tl_ag_gemm(ctypes.byref(a), _stream(stream)))


def tl_gemm_rs_workspace_size(R, M, N):
    return int(lib.tl_gemm_rs_workspace_size(R, M, N))


def tl_gemm_rs_num_flags(R, M, N):
    return int(lib.tl_gemm_rs_num_flags(R, M, N))


def tl_gemm_rs(A, B, out, workspace, signals: Signals, epoch: int, *, timeout_ns=0, trace=None, options=0,
               stream=None):
    """out[d] = rows d of sum_r A_r . B_r, rank order unless options say otherwise (see tilelink.h)."""
    R = len(A)
    M, K_r = A[0].shape
    N = B[0].shape[1]
    pa, pb, po = _ptr_array(A), _ptr_array(B), _ptr_array(out)
    a = tl_gemm_rs_args(R=R, M=M, K_r=K_r, N=N, A=ctypes.cast(pa, ctypes.POINTER(_vp)),
                        B=ctypes.cast(pb, ctypes.POINTER(_vp)), out=ctypes.cast(po, ctypes.POINTER(_vp)),
                        workspace=_ptr(workspace), workspace_bytes=workspace.numel() * workspace.element_size(),
                        signals=signals.handle, epoch=int(epoch) & 0xFFFFFFFF, options=int(options),
                        timeout_ns=int(timeout_ns), trace=_ptr(trace))
    _check(lib.tl_gemm_rs(ctypes.byref(a), _stream(stream)))


def tl_gemm_rs_noalloc(A, B, out, epoch: int, *, dev_status=None, timeout_ns=0, options=0, stream=None):
    """GEMM-RS for callers that cannot allocate device memory: the library's
    static device scratch replaces the workspace and the signals object.
    dev_status: optional int32 CUDA tensor of 4 words that receives device errors."""
    R = len(A)
    M, K_r = A[0].shape
    N = B[0].shape[1]
    pa, pb, po = _ptr_array(A), _ptr_array(B), _ptr_array(out)
    a = tl_gemm_rs_args(R=R, M=M, K_r=K_r, N=N, A=ctypes.cast(pa, ctypes.POINTER(_vp)),
                        B=ctypes.cast(pb, ctypes.POINTER(_vp)), out=ctypes.cast(po, ctypes.POINTER(_vp)),
                        workspace=None, workspace_bytes=0, signals=None, epoch=int(epoch) & 0xFFFFFFFF,
                        options=int(options), timeout_ns=int(timeout_ns), trace=None)
    _check(lib.tl_gemm_rs_noalloc(ctypes.byref(a), _ptr(dev_status), _stream(stream)))


def tl_moe_workspace_size(R, T_r, E, topk):
    return int(lib.tl_moe_workspace_size(R, T_r, E, topk))


def tl_moe_num_flags(R, T_r, H, topk, rows_per_barrier=0, mode=TL_MODE_PULL):
    eff = _i()
    n = lib.tl_moe_num_flags(mode, R, T_r, H, topk, rows_per_barrier, ctypes.byref(eff))
    return n, eff.value


def tl_moe_ag_gemm(X, topk_ids, W, sorted_tokens, Y, perm, expert_offsets, workspace, signals: Signals, epoch: int,
                   *, self_rank=0, rows_per_barrier=0, mode=TL_MODE_PULL, timeout_ns=0, trace=None, stream=None):
    """AllGather + grouped MoE GEMM (see tilelink.h): Y rows in expert-sorted order."""
    R = len(X)
    T_r, H = X[0].shape
    E = len(W)
    N = W[0].shape[1]
    topk = topk_ids.shape[1]
    px, pw = _ptr_array(X), _ptr_array(W)
    a = tl_moe_args(R=R, self_rank=self_rank, T_r=T_r, H=H, N=N, E=E, topk=topk, rows_per_barrier=rows_per_barrier,
                    X=ctypes.cast(px, ctypes.POINTER(_vp)), topk_ids=_ptr(topk_ids),
                    W=ctypes.cast(pw, ctypes.POINTER(_vp)), sorted_tokens=_ptr(sorted_tokens), Y=_ptr(Y),
                    perm=_ptr(perm), expert_offsets=_ptr(expert_offsets), workspace=_ptr(workspace),
                    workspace_bytes=workspace.numel() * workspace.element_size(), signals=signals.handle,
                    epoch=int(epoch) & 0xFFFFFFFF, mode=mode, timeout_ns=int(timeout_ns), trace=_ptr(trace))
    _check(lib.tl_moe_ag_gemm(ctypes.byref(a), _stream(stream)))


def tl_allgather(A_shards, gathered, signals: Signals, epoch: int, *, self_rank=0, mode=TL_MODE_PUSH,
                 src_ready: Signals | None = None, rows_per_barrier=0, timeout_ns=0, stream=None):
    """Gather the shards into `gathered`, releasing one flag per chunk (see tilelink.h)."""
    R = len(A_shards)
    M_shard, K = A_shards[0].shape
    ptrs = _ptr_array(A_shards)
    a = tl_allgather_args(R=R, self_rank=self_rank, M_shard=M_shard, K=K, mode=mode,
                          rows_per_barrier=rows_per_barrier, A_shards=ctypes.cast(ptrs, ctypes.POINTER(_vp)),
                          gathered=_ptr(gathered), signals=signals.handle,
                          src_ready=src_ready.handle if src_ready is not None else None,
                          epoch=int(epoch) & 0xFFFFFFFF, reserved0=0, timeout_ns=int(timeout_ns))
    _check(lib.tl_allgather(ctypes.byref(a), _stream(stream)))


def tl_allgather_ll_link_bytes(R, M_shard, K, rows_per_barrier=0):
    return int(lib.tl_allgather_ll_link_bytes(R, M_shard, K, rows_per_barrier))


def tl_allgather_ll(A_shards, link, gathered, signals: Signals, epoch: int, *, self_rank=0,
                    protocol=TL_LL_FLAG_IN_DATA, send_mask=None, rows_per_barrier=0, timeout_ns=0, stream=None):
    """AllGather through the link buffer `link` (pinned host or device tensor) with the
    flag-in-data protocol or the separate-flag one (see tilelink.h).  send_mask None =
    every rank sends in this launch."""
    R = len(A_shards)
    M_shard, K = A_shards[0].shape
    ptrs = _ptr_array(A_shards)
    mask = (1 << R) - 1 if send_mask is None else int(send_mask)
    a = tl_allgather_ll_args(R=R, self_rank=self_rank, M_shard=M_shard, K=K, protocol=int(protocol),
                             rows_per_barrier=rows_per_barrier, A_shards=ctypes.cast(ptrs, ctypes.POINTER(_vp)),
                             link=_ptr(link), link_bytes=_nbytes(link), gathered=_ptr(gathered),
                             signals=signals.handle, send_mask=mask, epoch=int(epoch) & 0xFFFFFFFF, reserved0=0,
                             timeout_ns=int(timeout_ns))
    _check(lib.tl_allgather_ll(ctypes.byref(a), _stream(stream)))


def tl_test_hold_chunks(first_flag, count, hold_ns):
    """Test facility: on this thread, later copy-warp calls move the chunks with flag ids in
    [first_flag, first_flag + count) last, after hold_ns (see tilelink.h).  count 0 = off."""
    _check(lib.tl_test_hold_chunks(int(first_flag), int(count), int(hold_ns)))


def tl_reduce_scatter(partials, out, *, stream=None):
    """out[d] = rows d of the rank-ordered fp32 sum of the partials, bf16."""
    R = len(partials)
    M, N = partials[0].shape
    pp, po = _ptr_array(partials), _ptr_array(out)
    a = tl_reduce_scatter_args(R=R, M=M, N=N, reserved0=0, partials=ctypes.cast(pp, ctypes.POINTER(_vp)),
                               out=ctypes.cast(po, ctypes.POINTER(_vp)))
    _check(lib.tl_reduce_scatter(ctypes.byref(a), _stream(stream)))


def tl_moe_down_workspace_size(R, T_r, topk, E, Hd):
    return int(lib.tl_moe_down_workspace_size(R, T_r, topk, E, Hd))


def tl_moe_down_num_flags(R, T_r, topk, E, Hd):
    return int(lib.tl_moe_down_num_flags(R, T_r, topk, E, Hd))


def tl_moe_down(H, W2, gates, routing, out, workspace, signals: Signals, epoch: int, *, topk, E, timeout_ns=0,
                options=0, stream=None):
    """out[d] = the gate-weighted combine of each token's expert outputs, Y summed over ranks
    (see tilelink.h); routing is the workspace of the matching tl_moe_ag_gemm call."""
    R = len(H)
    P, I_r = H[0].shape
    Hd = W2[0].shape[1]
    T_r = out[0].shape[0]
    ph, pw, po = _ptr_array(H), _ptr_array(W2), _ptr_array(out)
    a = tl_moe_down_args(R=R, T_r=T_r, topk=topk, E=E, I_r=I_r, Hd=Hd, H=ctypes.cast(ph, ctypes.POINTER(_vp)),
                         W2=ctypes.cast(pw, ctypes.POINTER(_vp)), gates=_ptr(gates), routing=_ptr(routing),
                         out=ctypes.cast(po, ctypes.POINTER(_vp)), workspace=_ptr(workspace),
                         workspace_bytes=workspace.numel() * workspace.element_size(), signals=signals.handle,
                         epoch=int(epoch) & 0xFFFFFFFF, options=int(options), timeout_ns=int(timeout_ns))
    _check(lib.tl_moe_down(ctypes.byref(a), _stream(stream)))


def tl_ag_attn_num_flags(R, S_shard):
    return int(lib.tl_ag_attn_num_flags(R, S_shard))


def tl_ag_attn(Q, K_shards, V_shards, K_gathered, V_gathered, O, signals: Signals, epoch: int, *, self_rank=0,
               causal=False, scale=0.0, lse=None, timeout_ns=0, stream=None):
    """O = softmax(scale Q Kg^T) Vg per head over the gathered key/value shards,
    K_gathered / V_gathered written (see tilelink.h).  Q [S_shard, H, D],
    K_r / V_r [S_shard, H_kv, D], lse optional float [H, S_shard]."""
    R = len(K_shards)
    S_shard, H, D = Q.shape
    H_kv = K_shards[0].shape[1]
    pk, pv = _ptr_array(K_shards), _ptr_array(V_shards)
    a = tl_ag_attn_args(R=R, self_rank=self_rank, S_shard=S_shard, H=H, H_kv=H_kv, head_dim=D,
                        causal=int(bool(causal)), scale=float(scale), Q=_ptr(Q),
                        K_shards=ctypes.cast(pk, ctypes.POINTER(_vp)), V_shards=ctypes.cast(pv, ctypes.POINTER(_vp)),
                        K_gathered=_ptr(K_gathered), V_gathered=_ptr(V_gathered), O=_ptr(O), lse=_ptr(lse),
                        signals=signals.handle, epoch=int(epoch) & 0xFFFFFFFF, reserved0=0,
                        timeout_ns=int(timeout_ns))
    _check(lib.tl_ag_attn(ctypes.byref(a), _stream(stream)))
