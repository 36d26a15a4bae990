"""ctypes binding of libkvc.so: the C ABI of include/kvc.h, same names.

Argument marshalling only: torch tensors are passed as device pointers, host
budget arrays as int32 arrays, the stream as the caller's current CUDA stream.
Every step of the compression runs in the library's CUDA kernels; there is no
other code path.  Importing this module fails loudly if the library has not
been built (``python -m attention_score_kv_gb300.build``).
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVC_LIBRARY selects another build of the same library (e.g. one compiled
# with different tuning flags); default: the in-tree libkvc.so.
LIB_PATH = os.environ.get("KVC_LIBRARY") or os.path.join(_HERE, "libkvc.so")

KVC_OK = 0
KVC_ERR_INVALID_ARG = -1
KVC_ERR_UNSUPPORTED = -2
KVC_ERR_WORKSPACE = -3
KVC_ERR_CUDA = -4
KVC_ERR_TIMEOUT = -5
KVC_ERR_DEVICE = -6
KVC_OPT_SCAN_CTAS = 1
KVC_OPT_WAIT_LIMIT = 2

_NAMES = {
    KVC_ERR_INVALID_ARG: "invalid argument", KVC_ERR_UNSUPPORTED: "unsupported",
    KVC_ERR_WORKSPACE: "workspace", KVC_ERR_CUDA: "CUDA", KVC_ERR_TIMEOUT: "timeout",
    KVC_ERR_DEVICE: "device status",
}


class KvcError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kvc error {code} ({_NAMES.get(code, '?')}): {msg}")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -m attention_score_kv_gb300.build` (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_I64 = ctypes.c_int64
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_F64P = ctypes.POINTER(ctypes.c_double)

_SIGS = {
    "kvc_last_error": (ctypes.c_char_p, []),
    "kvc_version": (_I, []),
    "kvc_workspace_size": (_SZ, [_I] * 8),
    "kvc_score_pass1": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "kvc_score_pass1_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "kvc_score_pass2_pool": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "kvc_score_rawdot_int8": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "kvc_select_topk": (_I, [_P, _I, _I, _I, _I32P, _I64P, _I, _I, _P, _P, _SZ, _P]),
    "kvc_gather": (_I, [_P, _P, _P, _I64P, _I, _I, _I, _I, _I32P, _P, _P, _P, _P]),
    "kvc_compress_layer": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I32P, _I, _I, _I, _I,
                                _P, _P, _P, _P, _P, _P, _I64P, _P, _SZ, _P]),
    "kvc_compress_layer_deferred_v": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I32P, _I, _I, _I, _I,
                                           _P, _P, _P, _P, _P, _P, _I64P, _P, _SZ, _P, _P]),
    "kvc_overlap_coefficient": (_I, [_P, _P, _P, _P, _I, _P, _P]),
    "kvc_head_similarity": (_I, [_P, _P, _I, _I, _P, _P]),
    "kvc_budget_inverse_stability_device": (_I, [_I, _I, _P, _I64, _I, _I, _P, _P]),
    "kvc_median_over_steps": (_I, [_P, _I, _I, _P, _P]),
    "kvc_head_stability_over_steps": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _P]),
    "kvc_head_similarity_over_steps": (_I, [_P, _P, _I, _I, _P, _P, _P]),
    "kvc_append_chunk": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "kvc_cache_layout": (_I, [_I, _I, _I, _I, _I32P, _I64P]),
    "kvc_scan_ranges": (_I, [_I, _I, _I, _I64P]),
    "kvc_budget_pyramid": (_I, [_I, _I, _I, _I32P]),
    "kvc_retained_layout": (_I, [_I, _I, _I32P, _I64P]),
    "kvc_budget_inverse_stability": (_I, [_I, _F64P, _I64, _I, _I, _I32P]),
    "kvc_check_status": (_I, [_P]),
    "kvc_set_option": (_I, [_I, _I64]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def lib() -> ctypes.CDLL:
    return _lib


def _check(rc: int) -> None:
    if rc != KVC_OK:
        raise KvcError(rc, _lib.kvc_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32(arr):
    vals = [int(x) for x in (arr.tolist() if hasattr(arr, "tolist") else arr)]
    return (ctypes.c_int32 * len(vals))(*vals)


def _i64_or_null(arr):
    """A host int64 array, or NULL for None (the packed output layout)."""
    if arr is None:
        return None
    vals = [int(x) for x in (arr.tolist() if hasattr(arr, "tolist") else arr)]
    return (ctypes.c_int64 * len(vals))(*vals)


def kvc_last_error() -> str:
    return _lib.kvc_last_error().decode()


def kvc_version() -> int:
    return _lib.kvc_version()


def kvc_workspace_size(B, H_q, H_kv, D, W, b_s, K_l_max, pool_k) -> int:
    n = _lib.kvc_workspace_size(B, H_q, H_kv, D, W, b_s, K_l_max, pool_k)
    if n == 0:
        raise KvcError(KVC_ERR_INVALID_ARG, kvc_last_error())
    return n


def kvc_score_pass1(q_win, k, B, H_q, H_kv, S, D, W, b_s, m, Z, ws, ws_bytes=None, stream=None):
    _check(_lib.kvc_score_pass1(_ptr(q_win), _ptr(k), B, H_q, H_kv, S, D, W, b_s, _ptr(m), _ptr(Z),
                                _ptr(ws), ws.numel() if ws_bytes is None else ws_bytes, _stream(stream)))


def kvc_score_pass1_noalloc(q_win, k, B, H_q, H_kv, S, D, W, b_s, m, Z, stream=None):
    """Pass 1 with the library's fixed scratch array instead of a workspace,
    for callers that may not allocate device memory (see include/kvc.h)."""
    _check(_lib.kvc_score_pass1_noalloc(_ptr(q_win), _ptr(k), B, H_q, H_kv, S, D, W, b_s, _ptr(m), _ptr(Z),
                                        _stream(stream)))


def kvc_score_pass2_pool(q_win, k, m, Z, B, H_q, H_kv, S, D, W, b_s, pool_k, scores, ws, ws_bytes=None,
                         stream=None):
    _check(_lib.kvc_score_pass2_pool(_ptr(q_win), _ptr(k), _ptr(m), _ptr(Z), B, H_q, H_kv, S, D, W, b_s,
                                     pool_k, _ptr(scores), _ptr(ws), ws.numel() if ws_bytes is None else ws_bytes,
                                     _stream(stream)))


def kvc_score_rawdot_int8(q_win, k, B, H_q, H_kv, S, D, W, scores, ws, ws_bytes=None, stream=None):
    _check(_lib.kvc_score_rawdot_int8(_ptr(q_win), _ptr(k), B, H_q, H_kv, S, D, W, _ptr(scores), _ptr(ws),
                                      ws.numel() if ws_bytes is None else ws_bytes, _stream(stream)))


def kvc_append_chunk(k_chunk, v_chunk, B, H_kv, S, C, D, j, k_act, v_act, stream=None):
    _check(_lib.kvc_append_chunk(_ptr(k_chunk), _ptr(v_chunk), B, H_kv, S, C, D, j, _ptr(k_act), _ptr(v_act),
                                 _stream(stream)))


def kvc_budget_pyramid(N, budget, k_min):
    out = (ctypes.c_int32 * N)()
    _check(_lib.kvc_budget_pyramid(N, budget, k_min, out))
    return list(out)


def kvc_cache_layout(N, B, H_kv, S, K_l):
    """Row offsets [N + 1] of each layer in the cross-layer retained cache."""
    flat = [int(x) for row in K_l for x in row]
    out = (ctypes.c_int64 * (N + 1))()
    _check(_lib.kvc_cache_layout(N, B, H_kv, S, _i32(flat), out))
    return list(out)


def kvc_overlap_coefficient(a, a_off, b, b_off, n_pairs, out, stream=None):
    _check(_lib.kvc_overlap_coefficient(_ptr(a), _ptr(a_off), _ptr(b), _ptr(b_off), n_pairs, _ptr(out),
                                        _stream(stream)))


def kvc_head_similarity(idx, off, n_groups, H, sim, stream=None):
    _check(_lib.kvc_head_similarity(_ptr(idx), _ptr(off), n_groups, H, _ptr(sim), _stream(stream)))


def kvc_median_over_steps(x, T, H, med, stream=None):
    _check(_lib.kvc_median_over_steps(_ptr(x), T, H, _ptr(med), _stream(stream)))


def kvc_head_stability_over_steps(dec_idx, dec_off, pre_idx, pre_off, T, H, per_step, stability, stream=None):
    _check(_lib.kvc_head_stability_over_steps(_ptr(dec_idx), _ptr(dec_off), _ptr(pre_idx), _ptr(pre_off), T, H,
                                              _ptr(per_step), _ptr(stability), _stream(stream)))


def kvc_head_similarity_over_steps(idx, off, T, H, per_step, similarity, stream=None):
    _check(_lib.kvc_head_similarity_over_steps(_ptr(idx), _ptr(off), T, H, _ptr(per_step), _ptr(similarity),
                                               _stream(stream)))


def kvc_budget_inverse_stability_device(n_layers, H_kv, s_stable, total, lo, hi, K_l_out, stream=None):
    _check(_lib.kvc_budget_inverse_stability_device(n_layers, H_kv, _ptr(s_stable), total, lo, hi, _ptr(K_l_out),
                                                    _stream(stream)))


def kvc_select_topk(scores, B, H_kv, S, K_l, sink, recent, idx, ws, ws_bytes=None, stream=None, out_off=None):
    _check(_lib.kvc_select_topk(_ptr(scores), B, H_kv, S, _i32(K_l), _i64_or_null(out_off), sink, recent, _ptr(idx),
                                _ptr(ws), ws.numel() if ws_bytes is None else ws_bytes, _stream(stream)))


def kvc_gather(k, v, idx, B, H_kv, S, D, K_l, k_out, v_out, pos_out, stream=None, out_off=None):
    _check(_lib.kvc_gather(_ptr(k), _ptr(v), _ptr(idx), _i64_or_null(out_off), B, H_kv, S, D, _i32(K_l),
                           _ptr(k_out), _ptr(v_out), _ptr(pos_out), _stream(stream)))


def kvc_compress_layer(N, layer, B, S, C, H_q, H_kv, D, W, K_l, sink, recent, pool_k, b_s, q_win, k, v,
                       k_out, v_out, pos_out, ws, ws_bytes=None, stream=None, out_off=None):
    _check(_lib.kvc_compress_layer(N, layer, B, S, C, H_q, H_kv, D, W, _i32(K_l), sink, recent, pool_k, b_s,
                                   _ptr(q_win), _ptr(k), _ptr(v), _ptr(k_out), _ptr(v_out), _ptr(pos_out),
                                   _i64_or_null(out_off), _ptr(ws), ws.numel() if ws_bytes is None else ws_bytes,
                                   _stream(stream)))


def _event(ev) -> int | None:
    if ev is None or isinstance(ev, int):
        return ev
    return ev.cuda_event   # torch.cuda.Event: its cudaEvent_t (0 until first recorded)


def kvc_compress_layer_deferred_v(N, layer, B, S, C, H_q, H_kv, D, W, K_l, sink, recent, pool_k, b_s, q_win, k, v,
                                  k_out, v_out, pos_out, ws, v_ready, ws_bytes=None, stream=None, out_off=None):
    """kvc_compress_layer whose gather first waits on the event v_ready
    (e.g. recorded after v's host-to-device copy on another stream)."""
    _check(_lib.kvc_compress_layer_deferred_v(N, layer, B, S, C, H_q, H_kv, D, W, _i32(K_l), sink, recent, pool_k,
                                              b_s, _ptr(q_win), _ptr(k), _ptr(v), _ptr(k_out), _ptr(v_out),
                                              _ptr(pos_out), _i64_or_null(out_off), _ptr(ws),
                                              ws.numel() if ws_bytes is None else ws_bytes, _event(v_ready),
                                              _stream(stream)))


def kvc_scan_ranges(BH, S, P) -> list:
    """Starts of the scan CTAs' key ranges over the flattened [BH][S] keys
    when P CTAs are asked for (the last entry is BH * S)."""
    out = (ctypes.c_int64 * (P + 1))()
    n = _lib.kvc_scan_ranges(BH, S, P, out)
    _check(min(n, 0))
    return list(out[:n + 1])


def kvc_retained_layout(H_kv, S, K_l) -> list:
    out = (ctypes.c_int64 * (H_kv + 1))()
    _check(_lib.kvc_retained_layout(H_kv, S, _i32(K_l), out))
    return list(out)


def kvc_budget_inverse_stability(s_stable, total, lo, hi) -> list:
    vals = [float(x) for x in (s_stable.tolist() if hasattr(s_stable, "tolist") else s_stable)]
    arr = (ctypes.c_double * len(vals))(*vals)
    out = (ctypes.c_int32 * len(vals))()
    _check(_lib.kvc_budget_inverse_stability(len(vals), arr, int(total), lo, hi, out))
    return list(out)


def kvc_check_status(stream=None) -> None:
    _check(_lib.kvc_check_status(_stream(stream)))


def kvc_set_option(option, value) -> None:
    _check(_lib.kvc_set_option(option, int(value)))


# ---------------------------------------------------------------- helpers
def workspace(B, H_q, H_kv, D, W, b_s, K_l_max, pool_k, device="cuda") -> torch.Tensor:
    """A uint8 device buffer of kvc_workspace_size(...) bytes (256-byte aligned)."""
    n = kvc_workspace_size(B, H_q, H_kv, D, W, b_s, K_l_max, pool_k)
    return torch.empty(n, dtype=torch.uint8, device=device)


def retained_outputs(B, H_kv, S, D, K_l, device="cuda"):
    """Allocate (k_out, v_out, pos_out, offsets) for the retained cache."""
    off = kvc_retained_layout(H_kv, S, K_l)
    T = off[-1]
    k_out = torch.empty((B * T, D), dtype=torch.bfloat16, device=device)
    v_out = torch.empty((B * T, D), dtype=torch.bfloat16, device=device)
    pos = torch.empty((B * T,), dtype=torch.int32, device=device)
    return k_out, v_out, pos, off


# ---------------------------------------------------------------- profiling
_lib.kvc_profile_begin.restype = _I
_lib.kvc_profile_begin.argtypes = []
_lib.kvc_profile_end.restype = _I
_lib.kvc_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), _I64P, _I64P]
KVC_N_STAGES = 4
STAGE_NAMES = ("pass1", "pass2_pool", "select_topk", "gather")
EXPORTED = EXPORTED + ("kvc_profile_begin", "kvc_profile_end")


def kvc_profile_begin() -> None:
    _check(_lib.kvc_profile_begin())


def kvc_profile_end():
    """Returns (stage_ms list, calls, launches) since kvc_profile_begin()."""
    ms = (ctypes.c_double * KVC_N_STAGES)()
    calls = ctypes.c_int64()
    launches = ctypes.c_int64()
    _check(_lib.kvc_profile_end(ms, ctypes.byref(calls), ctypes.byref(launches)))
    return list(ms), calls.value, launches.value
