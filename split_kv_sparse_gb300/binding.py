"""ctypes binding of ``include/mla_split.h`` (argument marshalling only).

Every function has the name of the C entry point it calls and does nothing but
convert arguments (torch tensors -> device pointers, streams -> handles) and
turn a non-zero status into ``SplitKVError``. All computation happens in the
CUDA library; there is no fallback: if ``libsplitkv.so`` is missing the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsplitkv.so")

MLA_OK = 0
MLA_OUT_F32, MLA_OUT_BF16, MLA_OUT_E4M3 = 0, 1, 2
MLA_STATUS_TIMEOUT = 0x1
MLA_STATUS_BAD_SHAPE = 0x2
MLA_STATUS_BAD_INDEX = 0x10
MLA_STATUS_BAD_ALIGN = 0x4
MLA_MAX_SPLITS = 64
MLA_FORCE_BALANCED = -1
OUT_DTYPES = {"f32": MLA_OUT_F32, "bf16": MLA_OUT_BF16, "e4m3": MLA_OUT_E4M3}

# Every symbol the header declares (checked by the library-load test).
EXPORTS = [
    "mla_decode_plan", "mla_sparse_decode_split", "mla_split_combine", "mla_sparse_decode_direct",
    "mla_sparse_decode", "mla_sparse_decode_host", "sdpa_fp8_decode_plan", "sdpa_fp8_decode_split",
    "sdpa_split_combine", "sdpa_fp8_decode_direct", "sdpa_fp8_decode", "mla_get_status",
    "mla_selftest_wait_timeout", "mla_status_string", "mla_abi_version", "mla_sparse_decode_noalloc",
    "mla_workspace_init", "mla_set_wait_limit_ns", "mla_plan_set_partials_bf16", "mla_set_index_checks",
]


class SplitKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


class MlaPlan(ctypes.Structure):
    _fields_ = [("s_q_max", ctypes.c_int32), ("h_q", ctypes.c_int32), ("d_qk", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("topk", ctypes.c_int32), ("block_rows", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("balanced_ctas", ctypes.c_int32), ("dim_groups", ctypes.c_int32),
                ("partial_bf16", ctypes.c_int32), ("tail_ctas", ctypes.c_int32), ("o_acc_bytes", ctypes.c_uint64),
                ("lse_acc_offset", ctypes.c_uint64), ("lse_acc_bytes", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64)]


class SdpaPlan(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("max_q_per_seq", ctypes.c_int32), ("total_q_max", ctypes.c_int32),
                ("max_kv", ctypes.c_int32), ("key_tile", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("adaptive_splits", ctypes.c_int32), ("o_acc_bytes", ctypes.c_uint64),
                ("lse_acc_offset", ctypes.c_uint64), ("lse_acc_bytes", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64

_SIGS = {
    "mla_decode_plan": [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(MlaPlan)],
    "mla_sparse_decode_split": [ctypes.POINTER(MlaPlan), _I, _P, _P, _I64, _P, _F, _P, _P],
    "mla_split_combine": [ctypes.POINTER(MlaPlan), _I, _P, _P, _I, _F, _P, _P, _P, _P],
    "mla_sparse_decode_direct": [_I, _I, _P, _P, _I64, _P, _F, _P, _I, _F, _P, _P, _P, _P],
    "mla_sparse_decode": [ctypes.POINTER(MlaPlan), _I, _P, _P, _I64, _P, _F, _P, _I, _F, _P, _P, _P, _P, _P],
    "mla_sparse_decode_host": [ctypes.POINTER(MlaPlan), _I, _P, _P, _P, _I64, _P, _P, _F, _P, _I, _F, _P, _P, _P,
                               _P, _P, _P, _P],
    "sdpa_fp8_decode_plan": [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(SdpaPlan)],
    "sdpa_fp8_decode_split": [ctypes.POINTER(SdpaPlan), _I, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P],
    "sdpa_split_combine": [ctypes.POINTER(SdpaPlan), _I, _P, _I, _F, _P, _P, _P, _P],
    "sdpa_fp8_decode_direct": [_I, _I, _I, _I, _I, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _F, _P, _P, _P,
                               _P],
    "sdpa_fp8_decode": [ctypes.POINTER(SdpaPlan), _I, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _F, _P, _P,
                        _P, _P, _P],
    "mla_get_status": [ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)],
    "mla_selftest_wait_timeout": [_U64, _P],
    "mla_status_string": [_I],
    "mla_abi_version": [],
    "mla_sparse_decode_noalloc": [_I, _I, _P, _P, _I64, _P, _F, _P, _I, _I, _F, _P, _P, _P, _P],
    "mla_workspace_init": [ctypes.POINTER(MlaPlan), _P, _P],
    "mla_set_wait_limit_ns": [_U64],
    "mla_set_index_checks": [_I],
    "mla_plan_set_partials_bf16": [ctypes.POINTER(MlaPlan), _I],
}


def lib() -> ctypes.CDLL:
    """Load libsplitkv.so (built in-tree by split_kv_sparse_gb300.build); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m split_kv_sparse_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name == "mla_status_string" else ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str):
    if st != MLA_OK:
        raise SplitKVError(st, where)


def _dtype(out_dtype) -> int:
    return OUT_DTYPES[out_dtype] if isinstance(out_dtype, str) else int(out_dtype)


# ---------------------------------------------------------------------- MLA --

def mla_decode_plan(s_q_max: int, topk: int, *, h_q: int = 64, d_qk: int = 576, d_v: int = 512,
                    num_sms: int = 0, max_splits: int = 0, force_splits: int = 0) -> MlaPlan:
    plan = MlaPlan()
    _check(lib().mla_decode_plan(s_q_max, h_q, d_qk, d_v, topk, num_sms, max_splits, force_splits,
                                 ctypes.byref(plan)), "mla_decode_plan")
    return plan


def mla_plan_set_partials_bf16(plan: MlaPlan, enable: bool = True) -> MlaPlan:
    """Switches the plan's O partials to bf16 (or back to fp32) in place; returns the plan."""
    _check(lib().mla_plan_set_partials_bf16(ctypes.byref(plan), enable if isinstance(enable, int) else int(enable)),
           "mla_plan_set_partials_bf16")
    return plan


def mla_workspace_init(plan: MlaPlan, workspace, stream=None):
    _check(lib().mla_workspace_init(ctypes.byref(plan), _ptr(workspace), _stream(stream)), "mla_workspace_init")


def mla_sparse_decode_split(plan: MlaPlan, s_q: int, q, kv, n_kv: int, idx, sm_scale: float, workspace,
                            stream=None):
    _check(lib().mla_sparse_decode_split(ctypes.byref(plan), s_q, _ptr(q), _ptr(kv), n_kv, _ptr(idx),
                                         sm_scale, _ptr(workspace), _stream(stream)),
           "mla_sparse_decode_split")


def mla_split_combine(plan: MlaPlan, s_q: int, workspace, sink, out_dtype, out_inv_scale: float, out,
                      lse_out=None, amax_out=None, stream=None):
    _check(lib().mla_split_combine(ctypes.byref(plan), s_q, _ptr(workspace), _ptr(sink), _dtype(out_dtype),
                                   out_inv_scale, _ptr(out), _ptr(lse_out), _ptr(amax_out), _stream(stream)),
           "mla_split_combine")


def mla_sparse_decode_direct(s_q: int, topk: int, q, kv, n_kv: int, idx, sm_scale: float, sink, out_dtype,
                             out_inv_scale: float, out, lse_out=None, amax_out=None, stream=None):
    _check(lib().mla_sparse_decode_direct(s_q, topk, _ptr(q), _ptr(kv), n_kv, _ptr(idx), sm_scale, _ptr(sink),
                                          _dtype(out_dtype), out_inv_scale, _ptr(out), _ptr(lse_out),
                                          _ptr(amax_out), _stream(stream)),
           "mla_sparse_decode_direct")


def mla_sparse_decode(plan: MlaPlan, s_q: int, q, kv, n_kv: int, idx, sm_scale: float, sink, out_dtype,
                      out_inv_scale: float, out, lse_out=None, amax_out=None, workspace=None, stream=None):
    _check(lib().mla_sparse_decode(ctypes.byref(plan), s_q, _ptr(q), _ptr(kv), n_kv, _ptr(idx), sm_scale,
                                   _ptr(sink), _dtype(out_dtype), out_inv_scale, _ptr(out), _ptr(lse_out),
                                   _ptr(amax_out), _ptr(workspace), _stream(stream)),
           "mla_sparse_decode")


def mla_sparse_decode_host(plan: MlaPlan, s_q: int, q_host, q_dev, kv, n_kv: int, idx_host, idx_dev,
                           sm_scale: float, sink, out_dtype, out_inv_scale: float, out_dev, out_host,
                           lse_dev=None, lse_host=None, amax_out=None, workspace=None, stream=None):
    """The decode step with q / idx / out / lse in host memory (pinned for asynchronous copies): the
    library copies them through the given device buffers around mla_sparse_decode, on `stream`."""
    _check(lib().mla_sparse_decode_host(ctypes.byref(plan), s_q, _ptr(q_host), _ptr(q_dev), _ptr(kv), n_kv,
                                        _ptr(idx_host), _ptr(idx_dev), sm_scale, _ptr(sink), _dtype(out_dtype),
                                        out_inv_scale, _ptr(out_dev), _ptr(out_host), _ptr(lse_dev),
                                        _ptr(lse_host), _ptr(amax_out), _ptr(workspace), _stream(stream)),
           "mla_sparse_decode_host")


# -------------------------------------------------------------------- dense --

def sdpa_fp8_decode_plan(batch: int, h_q: int, h_kv: int, d: int, max_q_per_seq: int, total_q_max: int,
                         max_kv: int, *, num_sms: int = 0, max_splits: int = 0, force_splits: int = 0) -> SdpaPlan:
    plan = SdpaPlan()
    _check(lib().sdpa_fp8_decode_plan(batch, h_q, h_kv, d, max_q_per_seq, total_q_max, max_kv, num_sms,
                                      max_splits, force_splits, ctypes.byref(plan)), "sdpa_fp8_decode_plan")
    return plan


def sdpa_fp8_decode_split(plan: SdpaPlan, total_q: int, total_kv: int, q, k, v, cu_seqlens_q, cu_seqlens_kv,
                          descale_q, descale_k, descale_v, sm_scale: float, workspace, stream=None):
    _check(lib().sdpa_fp8_decode_split(ctypes.byref(plan), total_q, total_kv, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(descale_q), _ptr(descale_k),
                                       _ptr(descale_v), sm_scale, _ptr(workspace), _stream(stream)),
           "sdpa_fp8_decode_split")


def sdpa_split_combine(plan: SdpaPlan, total_q: int, workspace, out_dtype, out_inv_scale: float, out,
                       lse_out=None, amax_out=None, stream=None):
    _check(lib().sdpa_split_combine(ctypes.byref(plan), total_q, _ptr(workspace), _dtype(out_dtype),
                                    out_inv_scale, _ptr(out), _ptr(lse_out), _ptr(amax_out), _stream(stream)),
           "sdpa_split_combine")


def sdpa_fp8_decode_direct(batch: int, h_q: int, h_kv: int, d: int, total_q: int, total_kv: int, q, k, v,
                           cu_seqlens_q, cu_seqlens_kv, descale_q, descale_k, descale_v, sm_scale: float, out_dtype,
                           out_inv_scale: float, out, lse_out=None, amax_out=None, stream=None):
    _check(lib().sdpa_fp8_decode_direct(batch, h_q, h_kv, d, total_q, total_kv, _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(descale_q),
                                        _ptr(descale_k), _ptr(descale_v), sm_scale, _dtype(out_dtype),
                                        out_inv_scale, _ptr(out), _ptr(lse_out), _ptr(amax_out), _stream(stream)),
           "sdpa_fp8_decode_direct")


def sdpa_fp8_decode(plan: SdpaPlan, total_q: int, total_kv: int, q, k, v, cu_seqlens_q, cu_seqlens_kv, descale_q,
                    descale_k, descale_v, sm_scale: float, out_dtype, out_inv_scale: float, out, lse_out=None,
                    amax_out=None, workspace=None, stream=None):
    _check(lib().sdpa_fp8_decode(ctypes.byref(plan), total_q, total_kv, _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_kv), _ptr(descale_q), _ptr(descale_k), _ptr(descale_v), sm_scale,
                                 _dtype(out_dtype), out_inv_scale, _ptr(out), _ptr(lse_out), _ptr(amax_out),
                                 _ptr(workspace), _stream(stream)),
           "sdpa_fp8_decode")


def mla_sparse_decode_noalloc(s_q: int, topk: int, q, kv, n_kv: int, idx, sm_scale: float, sink, num_splits: int,
                              out_dtype, out_inv_scale: float, out, lse_out=None, amax_out=None, stream=None):
    """Decode step whose split workspace is the library's own scratch array (no allocation)."""
    _check(lib().mla_sparse_decode_noalloc(s_q, topk, _ptr(q), _ptr(kv), n_kv, _ptr(idx), sm_scale, _ptr(sink),
                                           num_splits, _dtype(out_dtype), out_inv_scale, _ptr(out), _ptr(lse_out),
                                           _ptr(amax_out), _stream(stream)),
           "mla_sparse_decode_noalloc")


# ------------------------------------------------------------------- status --

def mla_get_status():
    """Synchronise the current device, then read and clear its status word: (bits, first site)."""
    st, site = ctypes.c_uint32(0), ctypes.c_uint32(0)
    _check(lib().mla_get_status(ctypes.byref(st), ctypes.byref(site)), "mla_get_status")
    return st.value, site.value


def mla_set_index_checks(enable: bool = True):
    """Report gathered indices outside {-1} and [0, n_kv) (status bit MLA_STATUS_BAD_INDEX) in later calls."""
    _check(lib().mla_set_index_checks(int(enable)), "mla_set_index_checks")


def mla_set_wait_limit_ns(limit_ns: int):
    """Time limit of the decode kernels' pipeline waits for later calls (0 = the 2 s default)."""
    _check(lib().mla_set_wait_limit_ns(limit_ns), "mla_set_wait_limit_ns")


def mla_selftest_wait_timeout(limit_ns: int, stream=None):
    _check(lib().mla_selftest_wait_timeout(limit_ns, _stream(stream)), "mla_selftest_wait_timeout")


def mla_abi_version() -> int:
    return lib().mla_abi_version()
