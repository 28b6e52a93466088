"""top_sparse_decode_gb300 -- Python binding of libsd (include/sd.h).

Every function has the name of the C entry point it calls and only marshals
arguments: tensors become device pointers, the stream defaults to torch's
current stream.  Every step of the path runs in libsd's CUDA kernels; there is
no Python or CPU fallback, and a missing libsd.so raises at first use.

bf16 tensors may be passed as torch.bfloat16 or as their int16/uint16 bit
patterns.  Layouts are those of include/sd.h (row-major, contiguous).
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _abi
from ._abi import (SD_ERR_CUDA, SD_ERR_INVALID_ARG, SD_ERR_TIMEOUT, SD_ERR_UNSUPPORTED,  # noqa: F401
                   SD_ERR_WORKSPACE, SD_IDX_LANDMARK, SD_IDX_MINMAX, SD_IDX_PLANES, SD_IDX_SIG,
                   SD_OK, SD_PLAN_FIXED, SD_PLAN_FULL, SD_PLAN_SPLIT, SD_PLAN_TOPQ,
                   SD_PLAN_WATERFILL,
                   SD_SCORE_F32, SD_SCORE_I32, SdEncoder, SdSelect, SdShape)

__all__ = [
    "SdError", "make_shape", "make_encoder", "make_select", "lib",
    "sd_build_index", "sd_append_index", "sd_encode_query", "sd_plan", "sd_score",
    "sd_topk_workspace_size", "sd_topk", "sd_gather_attend_workspace_size", "sd_gather_attend",
    "sd_gather_attend_noalloc", "sd_offload_gather", "Resident", "sd_delta_select",
    "sd_resident_gather",
    "sd_event_wait", "sd_last_error", "sd_version", "sd_launch_count", "sd_device_status",
    "sd_set_fallback_paths", "sd_debug_set_device_error", "sd_shard_candidates",
    "sd_topk_merge", "sd_shard_select", "sd_attend_combine",
    "sd_score_topk_workspace_size", "sd_score_topk", "sd_plan_score", "sd_topk_wmax", "sd_copy",
    "sd_select_attend_workspace_size", "sd_select_attend", "sd_hamming_topk_workspace_size",
    "sd_hamming_topk",
]


class SdError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def lib():
    return _abi.load()


def _check(rc: int, name: str) -> None:
    if rc != SD_OK:
        msg = (lib().sd_last_error() or b"").decode(errors="replace")
        raise SdError(rc, f"{name}: {msg}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("libsd takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_shape(batch: int, hq: int, hkv: int, n: int, d: int = 128, n_cap: int = 0) -> SdShape:
    return SdShape(batch, hq, hkv, d, n, n_cap)


class _Encoder:
    """sd_encoder plus references that keep its weight tensors alive."""

    def __init__(self, W1, b1=None, W2=None, b2=None):
        self.tensors = (W1, b1, W2, b2)
        hidden = 0 if W2 is None else int(W1.shape[0])
        self.c = SdEncoder(_ptr(W1), _ptr(b1), hidden, _ptr(W2), _ptr(b2))


def make_encoder(W1, b1=None, W2=None, b2=None) -> _Encoder:
    """Device fp32 weights: W1 [32][d] (single projection) or W1 [hidden][d] and
    W2 [32][hidden] (two layers)."""
    return _Encoder(W1, b1, W2, b2)


def make_select(k: int, sink: int = 0, local: int = 0, block: int = 1) -> SdSelect:
    return SdSelect(k, sink, local, block)


def sd_version() -> int:
    return int(lib().sd_version())


def sd_launch_count() -> int:
    return int(lib().sd_launch_count())


def sd_last_error() -> str:
    return (lib().sd_last_error() or b"").decode(errors="replace")


def sd_build_index(kind: int, shape: SdShape, K, enc: Optional[_Encoder], out0, out1=None,
                   stream=None) -> None:
    e = ctypes.byref(enc.c) if enc is not None else None
    _check(lib().sd_build_index(kind, ctypes.byref(shape), _ptr(K), e, _ptr(out0), _ptr(out1),
                                _stream(stream)), "sd_build_index")


def sd_append_index(kind: int, shape: SdShape, n_old: int, K, enc: Optional[_Encoder], out0,
                    out1=None, stream=None) -> None:
    e = ctypes.byref(enc.c) if enc is not None else None
    _check(lib().sd_append_index(kind, ctypes.byref(shape), n_old, _ptr(K), e, _ptr(out0),
                                 _ptr(out1), _stream(stream)), "sd_append_index")


def sd_encode_query(shape: SdShape, q, enc: _Encoder, qsig, stream=None) -> None:
    _check(lib().sd_encode_query(ctypes.byref(shape), _ptr(q), ctypes.byref(enc.c), _ptr(qsig),
                                 _stream(stream)), "sd_encode_query")


def sd_plan(shape: SdShape, q, sigma2, mode: int, budget: int, plan, stream=None) -> None:
    _check(lib().sd_plan(ctypes.byref(shape), _ptr(q), _ptr(sigma2), mode, budget, _ptr(plan),
                         _stream(stream)), "sd_plan")


def sd_score(kind: int, shape: SdShape, index0, index1, q_or_qsig, plan, scores,
             stream=None) -> None:
    _check(lib().sd_score(kind, ctypes.byref(shape), _ptr(index0), _ptr(index1),
                          _ptr(q_or_qsig), _ptr(plan), _ptr(scores), _stream(stream)),
           "sd_score")


def sd_topk_workspace_size(rows: int, n_units: int, sel: SdSelect) -> int:
    return int(lib().sd_topk_workspace_size(rows, n_units, ctypes.byref(sel)))


def sd_topk(score_type: int, scores, rows: int, n_units: int, n_tokens: int, sel: SdSelect,
            idx, idx_stride: int, count, workspace=None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sd_topk(score_type, _ptr(scores), rows, n_units, n_tokens, ctypes.byref(sel),
                         _ptr(idx), idx_stride, _ptr(count), _ptr(workspace), ws_bytes,
                         _stream(stream)), "sd_topk")


def sd_plan_score(shape: SdShape, planes, scales, q, sigma2, mode: int, budget: int, plan,
                  scores, wmax=None, stream=None) -> None:
    _check(lib().sd_plan_score(ctypes.byref(shape), _ptr(planes), _ptr(scales), _ptr(q),
                               _ptr(sigma2), mode, budget, _ptr(plan), _ptr(scores),
                               _ptr(wmax), _stream(stream)), "sd_plan_score")


def sd_topk_wmax(scores, wmax, rows: int, n: int, sel: SdSelect, idx, idx_stride: int, count,
                 workspace=None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sd_topk_wmax(_ptr(scores), _ptr(wmax), rows, n, ctypes.byref(sel), _ptr(idx),
                              idx_stride, _ptr(count), _ptr(workspace), ws_bytes,
                              _stream(stream)), "sd_topk_wmax")


def sd_hamming_topk_workspace_size(shape: SdShape, sel: SdSelect) -> int:
    return int(lib().sd_hamming_topk_workspace_size(ctypes.byref(shape), ctypes.byref(sel)))


def sd_hamming_topk(shape: SdShape, sig, qsig, sel: SdSelect, idx, idx_stride: int, count,
                    workspace=None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sd_hamming_topk(ctypes.byref(shape), _ptr(sig), _ptr(qsig), ctypes.byref(sel),
                                 _ptr(idx), idx_stride, _ptr(count), _ptr(workspace), ws_bytes,
                                 _stream(stream)), "sd_hamming_topk")


def sd_select_attend_workspace_size(shape: SdShape, sel: SdSelect, max_count: int) -> int:
    return int(lib().sd_select_attend_workspace_size(ctypes.byref(shape), ctypes.byref(sel),
                                                     max_count))


def sd_select_attend(shape: SdShape, scores, wmax, sel: SdSelect, q, K, V, scale: float, idx,
                     idx_stride: int, count, max_count: int, out, lse=None, workspace=None,
                     stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sd_select_attend(ctypes.byref(shape), _ptr(scores), _ptr(wmax),
                                  ctypes.byref(sel), _ptr(q), _ptr(K), _ptr(V), float(scale),
                                  _ptr(idx), idx_stride, _ptr(count), max_count, _ptr(out),
                                  _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)),
           "sd_select_attend")


def sd_score_topk_workspace_size(shape: SdShape, sel: SdSelect) -> int:
    return int(lib().sd_score_topk_workspace_size(ctypes.byref(shape), ctypes.byref(sel)))


def sd_score_topk(shape: SdShape, planes, scales, q, plan, sel: SdSelect, scores, idx,
                  idx_stride: int, count, workspace=None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sd_score_topk(ctypes.byref(shape), _ptr(planes), _ptr(scales), _ptr(q),
                               _ptr(plan), ctypes.byref(sel), _ptr(scores), _ptr(idx),
                               idx_stride, _ptr(count), _ptr(workspace), ws_bytes,
                               _stream(stream)), "sd_score_topk")


def sd_gather_attend_workspace_size(shape: SdShape, max_count: int) -> int:
    return int(lib().sd_gather_attend_workspace_size(ctypes.byref(shape), max_count))


def sd_gather_attend(shape: SdShape, q, K, V, idx, idx_stride: int, count, max_count: int,
                     scale: float, out, lse=None, workspace=None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sd_gather_attend(ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(V), _ptr(idx),
                                  idx_stride, _ptr(count), max_count, float(scale), _ptr(out),
                                  _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)),
           "sd_gather_attend")


def sd_gather_attend_noalloc(shape: SdShape, q, K, V, idx, idx_stride: int, count,
                             max_count: int, scale: float, out, lse=None, stream=None) -> None:
    """sd_gather_attend without a workspace (for callers that cannot allocate):
    partials live in libsd's 4 MiB per-GPU static array; see include/sd.h."""
    _check(lib().sd_gather_attend_noalloc(ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(V),
                                          _ptr(idx), idx_stride, _ptr(count), max_count,
                                          float(scale), _ptr(out), _ptr(lse), _stream(stream)),
           "sd_gather_attend_noalloc")


def sd_offload_gather(shape: SdShape, host_planes, host_scales, plan, dev_planes, dev_scales,
                      stream=None) -> None:
    _check(lib().sd_offload_gather(ctypes.byref(shape), _ptr(host_planes), _ptr(host_scales),
                                   _ptr(plan), _ptr(dev_planes), _ptr(dev_scales),
                                   _stream(stream)), "sd_offload_gather")


class Resident:
    """A resident set on the device (sd_resident): slot_unit and slot_last int32
    [rows][n_slots], unit_slot int32 [rows][n_units], all -1 when empty."""

    def __init__(self, rows: int, n_slots: int, n_units: int, device="cuda"):
        self.n_slots = n_slots
        self.slot_unit = torch.full((rows, n_slots), -1, dtype=torch.int32, device=device)
        self.slot_last = torch.full((rows, n_slots), -1, dtype=torch.int32, device=device)
        self.unit_slot = torch.full((rows, n_units), -1, dtype=torch.int32, device=device)
        self.c = _abi.SdResident(n_slots, _ptr(self.slot_unit), _ptr(self.slot_last),
                                 _ptr(self.unit_slot))


def sd_delta_select(shape: SdShape, sel: SdSelect, scores, idx, idx_stride: int, count,
                    admit_cap: int, step: int, res: Resident, plan_slot, plan_unit, plan_evict,
                    plan_count, pool_idx, pool_stride: int, pool_count, stream=None) -> None:
    _check(lib().sd_delta_select(ctypes.byref(shape), ctypes.byref(sel), _ptr(scores), _ptr(idx),
                                 idx_stride, _ptr(count), admit_cap, step, ctypes.byref(res.c),
                                 _ptr(plan_slot), _ptr(plan_unit), _ptr(plan_evict),
                                 _ptr(plan_count), _ptr(pool_idx), pool_stride, _ptr(pool_count),
                                 _stream(stream)), "sd_delta_select")


def sd_resident_gather(shape: SdShape, block: int, K, V, plan_slot, plan_unit, plan_count,
                       admit_cap: int, n_slots: int, K_pool, V_pool, stream=None) -> None:
    _check(lib().sd_resident_gather(ctypes.byref(shape), block, _ptr(K), _ptr(V), _ptr(plan_slot),
                                    _ptr(plan_unit), _ptr(plan_count), admit_cap, n_slots,
                                    _ptr(K_pool), _ptr(V_pool), _stream(stream)),
           "sd_resident_gather")


def sd_shard_candidates(scores, rows: int, n_s: int, idx, idx_stride: int, count, sink_s: int,
                        local_s: int, offset: int, k: int, cand_score, cand_idx, cand_count,
                        stream=None) -> None:
    _check(lib().sd_shard_candidates(_ptr(scores), rows, n_s, _ptr(idx), idx_stride, _ptr(count),
                                     sink_s, local_s, offset, k, _ptr(cand_score),
                                     _ptr(cand_idx), _ptr(cand_count), _stream(stream)),
           "sd_shard_candidates")


def sd_topk_merge(rows: int, shards: int, k: int, cand_score, cand_idx, cand_count, idx,
                  idx_stride: int, count, stream=None) -> None:
    _check(lib().sd_topk_merge(rows, shards, k, _ptr(cand_score), _ptr(cand_idx),
                               _ptr(cand_count), _ptr(idx), idx_stride, _ptr(count),
                               _stream(stream)), "sd_topk_merge")


def sd_shard_select(rows: int, sel_idx, sel_stride: int, sel_count, offset: int, n_s: int,
                    sink_s: int, local_s: int, k: int, idx, idx_stride: int, count,
                    stream=None) -> None:
    _check(lib().sd_shard_select(rows, _ptr(sel_idx), sel_stride, _ptr(sel_count), offset, n_s,
                                 sink_s, local_s, k, _ptr(idx), idx_stride, _ptr(count),
                                 _stream(stream)), "sd_shard_select")


def sd_attend_combine(shards: int, batch: int, hq: int, outs, lses, out, lse=None,
                      stream=None) -> None:
    _check(lib().sd_attend_combine(shards, batch, hq, _ptr(outs), _ptr(lses), _ptr(out),
                                   _ptr(lse), _stream(stream)), "sd_attend_combine")


def sd_device_status(stream=None) -> None:
    """Raises SdError(SD_ERR_TIMEOUT) when a kernel enqueued on `stream` (or earlier)
    stopped early because a bounded wait ran out; clears the report.  Waits for
    the stream."""
    _check(lib().sd_device_status(_stream(stream)), "sd_device_status")


def sd_set_fallback_paths(on: bool) -> bool:
    """Testing switch: route attention, top-k and the bit-plane scan to the kernels
    used where clusters cannot be co-resident (same results).  Returns the
    previous setting."""
    return bool(lib().sd_set_fallback_paths(1 if on else 0))


def sd_debug_set_device_error(stream=None) -> None:
    """Testing: raise the device error word that sd_device_status reports."""
    _check(lib().sd_debug_set_device_error(_stream(stream)), "sd_debug_set_device_error")


def sd_copy(dst, src, nbytes: Optional[int] = None, stream=None) -> None:
    """Kernel copy of nbytes (default: all of src) between device memory and pinned
    host memory (tensors or raw addresses)."""
    if nbytes is None:
        nbytes = src.numel() * src.element_size()
    _check(lib().sd_copy(_ptr(dst), _ptr(src), int(nbytes), _stream(stream)), "sd_copy")


def sd_event_wait(event, timeout_us: int) -> None:
    handle = event if isinstance(event, int) else event.cuda_event
    _check(lib().sd_event_wait(handle, int(timeout_us)), "sd_event_wait")


def default_scale(d: int = 128) -> float:
    """1/sqrt(d), the softmax scale of z_i = <q, k_i> / sqrt(d)."""
    return 1.0 / math.sqrt(d)
