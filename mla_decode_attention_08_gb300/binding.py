"""ctypes binding of libmla_decode (argument marshalling only).

Every function here forwards to the C ABI declared in ``include/mla_decode.h``
under the same name.  Tensors must already live on a CUDA device: there is no
CPU path, and a missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB as LIB_PATH

NUM_HEADS, QK_HEAD_DIM, V_HEAD_DIM, TILE_TOKENS = 16, 576, 512, 128

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported device", 3: "workspace too small",
          4: "CUDA call failed"}
DERR = {1: "qo_indptr", 2: "kv_indptr", 4: "kv_index", 8: "timeout", 16: "mx_scale"}


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, status)} (status {status})")
        self.status = status


class mla_plan_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_kv_len", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("abi_version", ctypes.c_int32),
                ("qo_len", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("ws_bytes", ctypes.c_uint64), ("ws_prefix_offset", ctypes.c_uint64),
                ("ws_workers_offset", ctypes.c_uint64), ("ws_lse_offset", ctypes.c_uint64),
                ("ws_partial_offset", ctypes.c_uint64)]


_VP, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_PLANP = ctypes.POINTER(mla_plan_t)
_FWD_ARGS = [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _PLANP, _VP, _I64, _I64, _VP, _SZ]
_FWD_BF16KV_ARGS = _FWD_ARGS[:2] + _FWD_ARGS[3:]  # no kv_scale
# q, kv_fp4, kv_scales, scale_bias, qo_indptr, kv_indptr, out, stream, plan, kv_rows, ws, ws_bytes
_FWD_MXFP4_ARGS = [_VP, _VP, _VP, _I32, _VP, _VP, _VP, _VP, _PLANP, _I64, _VP, _SZ]
SIGNATURES = {
    "mla_decode_plan": (ctypes.c_int, [_I32, _I32, _I32, _PLANP]),
    "mla_decode_plan_mtp": (ctypes.c_int, [_I32, _I32, _I32, _I32, _PLANP]),
    "mla_decode_fwd": (ctypes.c_int, _FWD_ARGS),
    "mla_decode_fwd_stall_stream": (ctypes.c_int, _FWD_ARGS),
    "mla_decode_stage1": (ctypes.c_int, _FWD_ARGS),
    "mla_decode_fwd_bf16kv": (ctypes.c_int, _FWD_BF16KV_ARGS),
    "mla_decode_stage1_bf16kv": (ctypes.c_int, _FWD_BF16KV_ARGS),
    "mla_decode_fwd_static_scratch": (ctypes.c_int, _FWD_ARGS[:-2]),
    "mla_decode_static_scratch_read_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _I32, _VP]),
    "mla_decode_fwd_mxfp4": (ctypes.c_int, _FWD_MXFP4_ARGS),
    "mla_decode_stage1_mxfp4": (ctypes.c_int, _FWD_MXFP4_ARGS),
    "mla_decode_fwd_mxfp4_stall_stream": (ctypes.c_int, _FWD_MXFP4_ARGS),
    "mla_mxfp4_quantize": (ctypes.c_int, [_VP, _I64, _VP, _VP, _VP]),
    "mla_debug_q_operand": (ctypes.c_int, [_VP, _I32, _I32, _VP, _VP, _VP, _VP]),
    "mla_decode_trace_read": (ctypes.c_int, [_VP, _VP, _I32]),
    "mla_debug_p_split": (ctypes.c_int, [_VP, _I64, _VP, _VP, _VP]),
    "mla_decode_stage2": (ctypes.c_int, [_VP, _VP, _VP, _PLANP, _VP, _SZ]),
    "mla_fp8_quantize_per_tensor": (ctypes.c_int, [_VP, _I64, _VP, _VP, _VP, _SZ, _VP]),
    "mla_decode_workspace_init": (ctypes.c_int, [_VP, _SZ, _VP]),
    "mla_decode_read_error": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_int32), _I32, _VP]),
    "mla_decode_schedule_host": (ctypes.c_int, [_VP, _I32, _I32, _VP, _VP]),
    "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mla_decode_abi_version": (ctypes.c_int32, []),
}

_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmla_decode.so (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(python -m mla_decode_attention_08_gb300.build)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name, None)
            if fn is None:  # a library from before this entry point; calling it raises
                continue
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MlaError(fn, status)


def _dev_ptr(t: Optional[torch.Tensor], name: str, dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def mla_decode_plan(batch: int, max_kv_len: int, num_sms: int = 0, qo_len: int = 1,
                    persistent: bool = False) -> mla_plan_t:
    """Plan for ``batch`` rows of ``qo_len`` query tokens (1 to 4; 2-4 for multi-token decode).

    ``persistent=True`` forces the persistent split (``plan.cluster = 0``) where
    the plan would take the cluster split of small batches."""
    plan = mla_plan_t()
    _check("mla_decode_plan_mtp", load_library().mla_decode_plan_mtp(batch, qo_len, max_kv_len,
                                                                    num_sms, ctypes.byref(plan)))
    if persistent:
        plan.cluster = 0
    return plan


def _e4m3_cache(kv_fp8) -> torch.Tensor:
    """The e4m3 cache as [rows, 576] bytes; anything else is refused (a bf16 or
    MXFP4 cache passed here would otherwise be read as e4m3 codes)."""
    if not isinstance(kv_fp8, torch.Tensor):
        raise TypeError("kv_fp8 must be a CUDA tensor")
    if kv_fp8.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"kv_fp8 must hold e4m3fn codes (uint8 or float8_e4m3fn), got {kv_fp8.dtype}")
    if kv_fp8.dim() not in (2, 3) or kv_fp8.numel() != kv_fp8.shape[0] * QK_HEAD_DIM:
        raise ValueError(f"kv_fp8 must be [rows, 576] or [rows, 1, 576], got {tuple(kv_fp8.shape)}")
    return kv_fp8.reshape(kv_fp8.shape[0], QK_HEAD_DIM)


def _fwd_args(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream, plan, kv_indices,
              workspace):
    kv_fp8 = _e4m3_cache(kv_fp8)
    kv_rows = int(kv_fp8.shape[0])
    return (_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(kv_fp8, "kv_fp8"),
            _dev_ptr(kv_scale, "kv_scale", torch.float32),
            _dev_ptr(qo_indptr, "qo_indptr", torch.int32),
            _dev_ptr(kv_indptr, "kv_indptr", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
            _stream(stream), ctypes.byref(plan),
            _dev_ptr(kv_indices, "kv_indices", torch.int32),
            0 if kv_indices is None else int(kv_indices.numel()), kv_rows,
            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size())


def _fwd_bf16kv_args(q, kv_bf16, qo_indptr, kv_indptr, out, stream, plan, kv_indices, workspace):
    if kv_bf16.dim() == 3:
        kv_bf16 = kv_bf16.reshape(kv_bf16.shape[0], -1)
    return (_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(kv_bf16, "kv_bf16", torch.bfloat16),
            _dev_ptr(qo_indptr, "qo_indptr", torch.int32),
            _dev_ptr(kv_indptr, "kv_indptr", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
            _stream(stream), ctypes.byref(plan),
            _dev_ptr(kv_indices, "kv_indices", torch.int32),
            0 if kv_indices is None else int(kv_indices.numel()), int(kv_bf16.shape[0]),
            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size())


def _fwd_mxfp4_args(q, kv_fp4, kv_scales, qo_indptr, kv_indptr, out, stream, plan, workspace,
                    scale_bias):
    kv_fp4 = kv_fp4.reshape(kv_fp4.shape[0], -1)
    if kv_fp4.shape[1] != QK_HEAD_DIM // 2 or kv_scales.numel() != kv_fp4.shape[0] * 18:
        raise ValueError("kv_fp4 must be [N, 288] uint8 and kv_scales [N, 18] uint8")
    return (_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(kv_fp4, "kv_fp4", torch.uint8),
            _dev_ptr(kv_scales, "kv_scales", torch.uint8), int(scale_bias),
            _dev_ptr(qo_indptr, "qo_indptr", torch.int32),
            _dev_ptr(kv_indptr, "kv_indptr", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
            _stream(stream), ctypes.byref(plan), int(kv_fp4.shape[0]),
            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size())


def mla_decode_fwd_mxfp4(q, kv_fp4, kv_scales, qo_indptr, kv_indptr, out, stream=None, *, plan,
                         workspace, scale_bias: int = 0) -> torch.Tensor:
    """Decode step over an MXFP4 cache (elements ``[N, 288]``, scales ``[N, 18]``); returns ``out``."""
    _check("mla_decode_fwd_mxfp4", load_library().mla_decode_fwd_mxfp4(
        *_fwd_mxfp4_args(q, kv_fp4, kv_scales, qo_indptr, kv_indptr, out, stream, plan, workspace,
                         scale_bias)))
    return out


def mla_decode_stage1_mxfp4(q, kv_fp4, kv_scales, qo_indptr, kv_indptr, out, stream=None, *,
                            plan, workspace, scale_bias: int = 0) -> None:
    _check("mla_decode_stage1_mxfp4", load_library().mla_decode_stage1_mxfp4(
        *_fwd_mxfp4_args(q, kv_fp4, kv_scales, qo_indptr, kv_indptr, out, stream, plan, workspace,
                         scale_bias)))


def mla_decode_fwd_mxfp4_stall_stream(q, kv_fp4, kv_scales, qo_indptr, kv_indptr, out,
                                      stream=None, *, plan, workspace, scale_bias: int = 0) -> None:
    """Test hook: the MXFP4 step with a cache stream that never arrives."""
    _check("mla_decode_fwd_mxfp4_stall_stream", load_library().mla_decode_fwd_mxfp4_stall_stream(
        *_fwd_mxfp4_args(q, kv_fp4, kv_scales, qo_indptr, kv_indptr, out, stream, plan, workspace,
                         scale_bias)))


def mla_mxfp4_quantize(src_bf16, dst_fp4, dst_scales, stream=None) -> None:
    """MXFP4 of bf16 rows ``[N, 576]`` into ``dst_fp4 [N, 288]`` and ``dst_scales [N, 18]``."""
    src = src_bf16.reshape(-1, QK_HEAD_DIM)
    rows = int(src.shape[0])
    if dst_fp4.numel() != rows * 288 or dst_scales.numel() != rows * 18:
        raise ValueError("dst_fp4 must hold [N, 288] and dst_scales [N, 18] bytes")
    _check("mla_mxfp4_quantize", load_library().mla_mxfp4_quantize(
        _dev_ptr(src, "src_bf16", torch.bfloat16), rows, _dev_ptr(dst_fp4, "dst_fp4", torch.uint8),
        _dev_ptr(dst_scales, "dst_scales", torch.uint8), _stream(stream)))


def mla_decode_fwd_bf16kv(q, kv_bf16, qo_indptr, kv_indptr, out, stream=None, *, plan,
                          workspace, kv_indices=None) -> torch.Tensor:
    """Decode step over a bf16 cache ``[N, 576]`` (no scale); writes and returns ``out``."""
    _check("mla_decode_fwd_bf16kv", load_library().mla_decode_fwd_bf16kv(
        *_fwd_bf16kv_args(q, kv_bf16, qo_indptr, kv_indptr, out, stream, plan, kv_indices,
                          workspace)))
    return out


def mla_decode_stage1_bf16kv(q, kv_bf16, qo_indptr, kv_indptr, out, stream=None, *, plan,
                             workspace, kv_indices=None) -> None:
    _check("mla_decode_stage1_bf16kv", load_library().mla_decode_stage1_bf16kv(
        *_fwd_bf16kv_args(q, kv_bf16, qo_indptr, kv_indptr, out, stream, plan, kv_indices,
                          workspace)))


def mla_decode_fwd(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream=None, *, plan,
                   workspace, kv_indices=None) -> torch.Tensor:
    """Decode step; writes ``out`` (bf16 [B, 16, 512]) and returns it."""
    _check("mla_decode_fwd", load_library().mla_decode_fwd(
        *_fwd_args(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream, plan, kv_indices,
                   workspace)))
    return out


def mla_decode_fwd_stall_stream(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream=None, *,
                                plan, workspace, kv_indices=None) -> None:
    """Test hook: the decode launches with a cache stream that never arrives,
    so the bounded waits run out and the call reports MLA_DERR_TIMEOUT."""
    _check("mla_decode_fwd_stall_stream", load_library().mla_decode_fwd_stall_stream(
        *_fwd_args(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream, plan, kv_indices,
                   workspace)))


def mla_decode_fwd_static_scratch(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream=None, *,
                                  plan, kv_indices=None) -> torch.Tensor:
    """Decode step with the library's own static scratch instead of a workspace,
    for callers that may not allocate device memory (see the C header)."""
    kv_fp8 = _e4m3_cache(kv_fp8)
    _check("mla_decode_fwd_static_scratch", load_library().mla_decode_fwd_static_scratch(
        _dev_ptr(q, "q", torch.bfloat16), _dev_ptr(kv_fp8, "kv_fp8"),
        _dev_ptr(kv_scale, "kv_scale", torch.float32), _dev_ptr(qo_indptr, "qo_indptr", torch.int32),
        _dev_ptr(kv_indptr, "kv_indptr", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
        _stream(stream), ctypes.byref(plan), _dev_ptr(kv_indices, "kv_indices", torch.int32),
        0 if kv_indices is None else int(kv_indices.numel()), int(kv_fp8.shape[0])))
    return out


def mla_decode_static_scratch_read_error(clear: bool = True, stream=None) -> int:
    """Error word of the current device's static scratch (MLA_DERR_* bits)."""
    v = ctypes.c_int32(0)
    _check("mla_decode_static_scratch_read_error",
           load_library().mla_decode_static_scratch_read_error(ctypes.byref(v), int(clear),
                                                               _stream(stream)))
    return int(v.value)


def mla_decode_stage1(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream=None, *, plan,
                      workspace, kv_indices=None) -> None:
    _check("mla_decode_stage1", load_library().mla_decode_stage1(
        *_fwd_args(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, out, stream, plan, kv_indices,
                   workspace)))


def mla_decode_stage2(qo_indptr, out, stream=None, *, plan, workspace) -> None:
    _check("mla_decode_stage2", load_library().mla_decode_stage2(
        _dev_ptr(qo_indptr, "qo_indptr", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
        _stream(stream), ctypes.byref(plan), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size()))


def mla_fp8_quantize_per_tensor(src_bf16, dst_fp8, scale_out, tmp, stream=None) -> None:
    """e4m3fn codes of a bf16 tensor with a per-tensor absmax scale (float32 [1])."""
    _check("mla_fp8_quantize_per_tensor", load_library().mla_fp8_quantize_per_tensor(
        _dev_ptr(src_bf16, "src", torch.bfloat16), src_bf16.numel(), _dev_ptr(dst_fp8, "dst"),
        _dev_ptr(scale_out, "scale_out", torch.float32), _dev_ptr(tmp, "tmp"),
        tmp.numel() * tmp.element_size(), _stream(stream)))


def mla_debug_q_operand(q, kv_scale, tokens_per_cta: int = 1, stream=None):
    """Test hook: stage 1's query operand of an e4m3 cache for every token of
    ``q`` [T, 16, 576]: (codes uint8 [T, 2, 16, 576] = hi then lo, qk_scale float [T])."""
    t = int(q.shape[0])
    codes = torch.empty((t, 2, NUM_HEADS, QK_HEAD_DIM), dtype=torch.uint8, device=q.device)
    qk_scale = torch.empty(t, dtype=torch.float32, device=q.device)
    _check("mla_debug_q_operand", load_library().mla_debug_q_operand(
        _dev_ptr(q, "q", torch.bfloat16), t, int(tokens_per_cta),
        _dev_ptr(kv_scale, "kv_scale", torch.float32), _dev_ptr(codes, "codes"),
        _dev_ptr(qk_scale, "qk_scale"), _stream(stream)))
    return codes, qk_scale


def mla_debug_p_split(p, stream=None):
    """Test hook: stage 1's two-term e4m3 split of float probabilities ``p``
    (numel a multiple of 16): (hi uint8, lo uint8), shaped like ``p``."""
    hi = torch.empty(p.shape, dtype=torch.uint8, device=p.device)
    lo = torch.empty(p.shape, dtype=torch.uint8, device=p.device)
    _check("mla_debug_p_split", load_library().mla_debug_p_split(
        _dev_ptr(p, "p", torch.float32), p.numel(), _dev_ptr(hi, "hi"), _dev_ptr(lo, "lo"),
        _stream(stream)))
    return hi, lo


TRACE_CTAS, TRACE_EVENTS, TRACE2_BLOCKS = 320, 40, 4096


def mla_decode_trace_read(clear: bool = True):
    """Trace builds only: (stage-1 stamps uint64 [TRACE_CTAS, TRACE_EVENTS], stage-2 stamps uint64 [TRACE2_BLOCKS, 3])."""
    import numpy as np
    s1 = np.zeros((TRACE_CTAS, TRACE_EVENTS), dtype=np.uint64)
    s2 = np.zeros((TRACE2_BLOCKS, 3), dtype=np.uint64)
    _check("mla_decode_trace_read", load_library().mla_decode_trace_read(
        s1.ctypes.data, s2.ctypes.data, int(clear)))
    return s1, s2


def mla_decode_workspace_init(workspace, stream=None) -> None:
    _check("mla_decode_workspace_init", load_library().mla_decode_workspace_init(
        _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def mla_decode_read_error(workspace, clear: bool = True, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("mla_decode_read_error", load_library().mla_decode_read_error(
        _dev_ptr(workspace, "workspace"), ctypes.byref(v), int(clear), _stream(stream)))
    return int(v.value)


def mla_decode_schedule_host(kv_indptr, grid: int):
    """(workers int32 [grid, 4], prefix int32 [B + 1]) from a host kv_indptr."""
    import numpy as np
    ind = np.ascontiguousarray(np.asarray(kv_indptr, dtype=np.int32))
    batch = ind.shape[0] - 1
    workers = np.zeros((grid, 4), dtype=np.int32)
    prefix = np.zeros(batch + 1, dtype=np.int32)
    _check("mla_decode_schedule_host", load_library().mla_decode_schedule_host(
        ind.ctypes.data, batch, grid, workers.ctypes.data, prefix.ctypes.data))
    return workers, prefix


def new_workspace(plan: mla_plan_t, device=None) -> torch.Tensor:
    """A zeroed uint8 workspace of plan.ws_bytes on ``device`` (256-byte aligned)."""
    ws = torch.zeros(int(plan.ws_bytes), dtype=torch.uint8, device=device or "cuda")
    assert ws.data_ptr() % 256 == 0
    return ws


def workspace_views(plan: mla_plan_t, ws: torch.Tensor) -> dict:
    """Typed views of the workspace regions (for tests and tools)."""
    g, b, nq = int(plan.grid), int(plan.batch), int(plan.qo_len)

    def view(off, n, dtype):
        size = torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + n * size].view(dtype)

    return {"err": view(0, 1, torch.int32),
            "prefix": view(plan.ws_prefix_offset, b + 1, torch.int32),
            "workers": view(plan.ws_workers_offset, 8 * g, torch.int32).view(g, 8)[:, :4],
            "jobs": view(plan.ws_workers_offset, 8 * g, torch.int32).view(g, 8)[:, 4:],
            "lse": view(plan.ws_lse_offset, 2 * g * nq * 16, torch.float32).view(2 * g, nq, 16),
            # bf16, stored [slot][token][dim / 128][head / 8][dim % 128][head % 8];
            # viewed as [slot][token][head][dim]
            "partial": view(plan.ws_partial_offset, 2 * g * nq * 16 * 512, torch.bfloat16)
                       .view(2 * g, nq, 4, 2, 128, 8).permute(0, 1, 3, 5, 2, 4)
                       .reshape(2 * g, nq, 16, 512)}
