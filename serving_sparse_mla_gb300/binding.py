"""Thin ctypes binding over the C ABI in include/sparse_mla.h.

Argument marshalling only: shape/dtype/device checks, raw pointers and sizes,
output allocation through torch.  Every step of the attention runs in the
CUDA library; there is no fallback.  Loading fails loudly when the library
has not been built.

The C ABI receives pointers and sizes only, so the extents are checked
here: every tensor a call reads or writes (inputs, caller-supplied outputs
and workspaces) must sit on the call's device and hold at least the
elements the passed sizes address, and caller-supplied outputs must have
the output's dtype and be contiguous; otherwise ValueError is raised before
anything is launched.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

_LIB: Optional[ctypes.CDLL] = None

c_int, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

STATUS = {0: "SPARSE_MLA_OK", 1: "SPARSE_MLA_ERR_INVALID_ARG", 2: "SPARSE_MLA_ERR_UNSUPPORTED_SHAPE",
          3: "SPARSE_MLA_ERR_UNSUPPORTED_ARCH", 4: "SPARSE_MLA_ERR_CUDA", 5: "SPARSE_MLA_ERR_DEVICE_TIMEOUT",
          6: "SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL"}

# name -> (restype, argtypes); the exported surface of include/sparse_mla.h
SIGNATURES = {
    "sparse_mla_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_float, c_void_p, c_void_p,
                               c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "sparse_mla_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_float,
                               c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "sparse_mla_bwd_varlen": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                      c_void_p, c_void_p, c_float, c_void_p, c_void_p, c_int, c_int, c_int,
                                      c_int, c_int, c_int, c_void_p]),
    "sparse_mla_fwd_causal": (c_int, [c_void_p, c_void_p, c_float, c_void_p, c_void_p,
                                      c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "sparse_mla_fwd_varlen": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_float,
                                      c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "sparse_mla_decode_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "sparse_mla_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_float, c_void_p,
                                  c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                  c_void_p, c_size_t, c_void_p]),
    "sparse_mla_decode_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_float, c_void_p,
                                      c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                      c_void_p, c_size_t, c_void_p]),
    "sparse_mla_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_float, c_void_p,
                                          c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                          c_void_p]),
    "sparse_mla_decode_noalloc_max_scratch_bytes": (c_size_t, []),
    "sparse_mla_debug_valid_count": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "sparse_mla_debug_valid_count_varlen": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                                    c_void_p, c_void_p]),
    "sparse_mla_debug_valid_count_paged": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                                   c_int, c_int, c_void_p, c_void_p]),
    "dsa_indexer_scores": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                   c_int, c_int, c_int, c_int, c_int, c_void_p, ctypes.c_longlong, c_void_p]),
    "dsa_topk": (c_int, [c_void_p, ctypes.c_longlong, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                         c_int, c_void_p, c_void_p]),
    "dsa_indexer_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "dsa_indexer_topk": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "dsa_indexer_scores_paged": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                         c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p,
                                         ctypes.c_longlong, c_void_p]),
    "dsa_indexer_topk_paged": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                       c_int, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_size_t,
                                       c_void_p]),
    "sparse_mla_status_string": (ctypes.c_char_p, [c_int]),
    "sparse_mla_get_device_error": (c_int, [ctypes.POINTER(c_int)]),
    "sparse_mla_clear_device_error": (c_int, []),
    "sparse_mla_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
}


class SparseMLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the built library (raises if it is missing)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise SparseMLAError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _on_cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _need(t: torch.Tensor, dtype, name: str):
    _on_cuda(t, name)
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _device_key(device):
    d = torch.device(device)
    if d.type == "cuda" and d.index is None:   # "cuda" means the current device
        return ("cuda", torch.cuda.current_device())
    return (d.type, d.index)


def _fits(t: Optional[torch.Tensor], need: int, name: str, device) -> None:
    """The kernels address t as a dense array of `need` elements on `device`.
    The C ABI sees only pointers and sizes, so extents are checked here: a
    tensor on another device, or with fewer elements than the sizes passed
    to the library imply, is refused before anything is launched."""
    if t is None:
        return
    if _device_key(t.device) != _device_key(device):
        raise ValueError(f"{name} is on {t.device}; the call's tensors are on {device}")
    if t.numel() < need:
        raise ValueError(f"{name} holds {t.numel()} elements; the call addresses {need}")


def _given(t: Optional[torch.Tensor], dtype, name: str, need: int, device) -> None:
    """A caller-supplied output or workspace: CUDA, dtype, contiguous, large
    enough and on the call's device."""
    if t is None:
        return
    _need(t, dtype, name)
    _fits(t, need, name, device)


def sparse_mla_fwd(q: torch.Tensor, kv: torch.Tensor, indices: torch.Tensor, sm_scale: float,
                   out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """q [s_q,h_q,576] bf16, kv [s_kv,576] or [s_kv,1,576] bf16,
    indices [s_q,topk] or [s_q,1,topk] int32 -> (out [s_q,h_q,512] bf16,
    lse [s_q,h_q] fp32)."""
    lib = load()
    s_q, h_q, d_qk = q.shape
    s_kv = kv.shape[0]
    topk = indices.shape[-1]
    for t, dt, n in ((q, torch.bfloat16, "q"), (kv, torch.bfloat16, "kv"), (indices, torch.int32, "indices")):
        _need(t, dt, n)
    d_v = 512
    dev = q.device
    _fits(kv, s_kv * d_qk, "kv", dev)
    _fits(indices, s_q * topk, "indices", dev)
    _given(out, torch.bfloat16, "out", s_q * h_q * d_v, dev)
    _given(lse, torch.float32, "lse", s_q * h_q, dev)
    if out is None:
        out = torch.empty((s_q, h_q, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    st = lib.sparse_mla_fwd(_ptr(q), _ptr(kv), _ptr(indices), float(sm_scale), _ptr(out), _ptr(lse),
                            s_q, s_kv, h_q, d_qk, d_v, topk, _stream(stream))
    _check(st, "sparse_mla_fwd")
    return out, lse


def sparse_mla_bwd(q: torch.Tensor, kv: torch.Tensor, indices: torch.Tensor, sm_scale: float,
                   out: torch.Tensor, lse: torch.Tensor, dout: torch.Tensor,
                   dq: Optional[torch.Tensor] = None, dkv: Optional[torch.Tensor] = None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Gradients of sparse_mla_fwd: q [s_q,h_q,576], kv [s_kv,576], indices
    [s_q,topk], the forward's out [s_q,h_q,512] bf16 and lse [s_q,h_q] fp32,
    dout [s_q,h_q,512] bf16 -> (dq [s_q,h_q,576] fp32, dkv [s_kv,576] fp32)."""
    lib = load()
    s_q, h_q, d_qk = q.shape
    s_kv = kv.shape[0]
    topk = indices.shape[-1]
    for t, dt, n in ((q, torch.bfloat16, "q"), (kv, torch.bfloat16, "kv"), (indices, torch.int32, "indices"),
                     (out, torch.bfloat16, "out"), (lse, torch.float32, "lse"), (dout, torch.bfloat16, "dout")):
        _need(t, dt, n)
    d_v = 512
    dev = q.device
    _fits(kv, s_kv * d_qk, "kv", dev)
    _fits(indices, s_q * topk, "indices", dev)
    _fits(out, s_q * h_q * d_v, "out", dev)
    _fits(lse, s_q * h_q, "lse", dev)
    _fits(dout, s_q * h_q * d_v, "dout", dev)
    _given(dq, torch.float32, "dq", s_q * h_q * d_qk, dev)
    _given(dkv, torch.float32, "dkv", s_kv * d_qk, dev)
    if dq is None:
        dq = torch.empty((s_q, h_q, d_qk), dtype=torch.float32, device=q.device)
    if dkv is None:
        dkv = torch.empty((s_kv, d_qk), dtype=torch.float32, device=q.device)
    st = lib.sparse_mla_bwd(_ptr(q), _ptr(kv), _ptr(indices), _ptr(out), _ptr(lse), _ptr(dout), float(sm_scale),
                            _ptr(dq), _ptr(dkv), s_q, s_kv, h_q, d_qk, d_v, topk, _stream(stream))
    _check(st, "sparse_mla_bwd")
    return dq, dkv


def sparse_mla_bwd_varlen(q, kv, indices, cu_seqlens_q, cu_seqlens_kv, sm_scale, out, lse, dout,
                          dq=None, dkv=None, stream=None):
    """Backward of sparse_mla_fwd_varlen -> (dq [total_q,h_q,576] fp32,
    dkv [total_kv,576] fp32)."""
    lib = load()
    total_q, h_q, d_qk = q.shape
    total_kv = kv.shape[0]
    topk = indices.shape[-1]
    batch = cu_seqlens_q.numel() - 1
    for t, dt, n in ((q, torch.bfloat16, "q"), (kv, torch.bfloat16, "kv"), (indices, torch.int32, "indices"),
                     (cu_seqlens_q, torch.int32, "cu_seqlens_q"), (cu_seqlens_kv, torch.int32, "cu_seqlens_kv"),
                     (out, torch.bfloat16, "out"), (lse, torch.float32, "lse"), (dout, torch.bfloat16, "dout")):
        _need(t, dt, n)
    dev = q.device
    _fits(kv, total_kv * d_qk, "kv", dev)
    _fits(indices, total_q * topk, "indices", dev)
    _fits(cu_seqlens_q, batch + 1, "cu_seqlens_q", dev)
    _fits(cu_seqlens_kv, batch + 1, "cu_seqlens_kv", dev)
    _fits(out, total_q * h_q * 512, "out", dev)
    _fits(lse, total_q * h_q, "lse", dev)
    _fits(dout, total_q * h_q * 512, "dout", dev)
    _given(dq, torch.float32, "dq", total_q * h_q * d_qk, dev)
    _given(dkv, torch.float32, "dkv", total_kv * d_qk, dev)
    if dq is None:
        dq = torch.empty((total_q, h_q, d_qk), dtype=torch.float32, device=q.device)
    if dkv is None:
        dkv = torch.empty((total_kv, d_qk), dtype=torch.float32, device=q.device)
    st = lib.sparse_mla_bwd_varlen(_ptr(q), _ptr(kv), _ptr(indices), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
                                   batch, _ptr(out), _ptr(lse), _ptr(dout), float(sm_scale), _ptr(dq), _ptr(dkv),
                                   total_q, total_kv, h_q, d_qk, 512, topk, _stream(stream))
    _check(st, "sparse_mla_bwd_varlen")
    return dq, dkv


def sparse_mla_fwd_causal(q: torch.Tensor, kv: torch.Tensor, sm_scale: float,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Indices-free causal forward: q [s_q,h_q,576] bf16 (the last s_q of the
    s_kv positions), kv [s_kv,576] or [s_kv,1,576] bf16 -> (out [s_q,h_q,512]
    bf16, lse [s_q,h_q] fp32)."""
    lib = load()
    s_q, h_q, d_qk = q.shape
    s_kv = kv.shape[0]
    for t, dt, n in ((q, torch.bfloat16, "q"), (kv, torch.bfloat16, "kv")):
        _need(t, dt, n)
    d_v = 512
    dev = q.device
    _fits(kv, s_kv * d_qk, "kv", dev)
    _given(out, torch.bfloat16, "out", s_q * h_q * d_v, dev)
    _given(lse, torch.float32, "lse", s_q * h_q, dev)
    if out is None:
        out = torch.empty((s_q, h_q, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    st = lib.sparse_mla_fwd_causal(_ptr(q), _ptr(kv), float(sm_scale), _ptr(out), _ptr(lse),
                                   s_q, s_kv, h_q, d_qk, d_v, _stream(stream))
    _check(st, "sparse_mla_fwd_causal")
    return out, lse


def sparse_mla_fwd_varlen(q, kv, indices, cu_seqlens_q, cu_seqlens_kv, sm_scale, out=None, lse=None,
                          stream=None):
    """Packed prefill; indices are local to each token's sequence."""
    lib = load()
    total_q, h_q, d_qk = q.shape
    total_kv = kv.shape[0]
    topk = indices.shape[-1]
    batch = cu_seqlens_q.numel() - 1
    for t, dt, n in ((q, torch.bfloat16, "q"), (kv, torch.bfloat16, "kv"), (indices, torch.int32, "indices"),
                     (cu_seqlens_q, torch.int32, "cu_seqlens_q"), (cu_seqlens_kv, torch.int32, "cu_seqlens_kv")):
        _need(t, dt, n)
    dev = q.device
    _fits(kv, total_kv * d_qk, "kv", dev)
    _fits(indices, total_q * topk, "indices", dev)
    _fits(cu_seqlens_q, batch + 1, "cu_seqlens_q", dev)
    _fits(cu_seqlens_kv, batch + 1, "cu_seqlens_kv", dev)
    _given(out, torch.bfloat16, "out", total_q * h_q * 512, dev)
    _given(lse, torch.float32, "lse", total_q * h_q, dev)
    if out is None:
        out = torch.empty((total_q, h_q, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((total_q, h_q), dtype=torch.float32, device=q.device)
    st = lib.sparse_mla_fwd_varlen(_ptr(q), _ptr(kv), _ptr(indices), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
                                   batch, float(sm_scale), _ptr(out), _ptr(lse), total_q, total_kv, h_q, d_qk,
                                   512, topk, _stream(stream))
    _check(st, "sparse_mla_fwd_varlen")
    return out, lse


def decode_workspace_size(batch: int, s_next: int, h_q: int, topk: int, d_v: int = 512) -> int:
    return int(load().sparse_mla_decode_workspace_size(batch, s_next, h_q, d_v, topk))


def sparse_mla_decode(q, kv_cache, block_table, cache_seqlens, indices, sm_scale, page_size=None,
                      workspace: Optional[torch.Tensor] = None, out=None, lse=None, stream=None):
    """Paged decode.  q [b,s_next,h_q,576]; kv_cache [num_blocks,page,576]
    (or [num_blocks,page,1,576]); block_table [b,max_blocks];
    cache_seqlens [b]; indices [b,s_next,topk] logical positions."""
    lib = load()
    batch, s_next, h_q, d_qk = q.shape
    num_blocks = kv_cache.shape[0]
    page = kv_cache.shape[1] if page_size is None else page_size
    max_blocks = block_table.shape[1]
    topk = indices.shape[-1]
    for t, dt, n in ((q, torch.bfloat16, "q"), (kv_cache, torch.bfloat16, "kv_cache"),
                     (block_table, torch.int32, "block_table"), (cache_seqlens, torch.int32, "cache_seqlens"),
                     (indices, torch.int32, "indices")):
        _need(t, dt, n)
    dev = q.device
    _fits(kv_cache, num_blocks * page * d_qk, "kv_cache", dev)
    _fits(block_table, batch * max_blocks, "block_table", dev)
    _fits(cache_seqlens, batch, "cache_seqlens", dev)
    _fits(indices, batch * s_next * topk, "indices", dev)
    _given(out, torch.bfloat16, "out", batch * s_next * h_q * 512, dev)
    _given(lse, torch.float32, "lse", batch * s_next * h_q, dev)
    _workspace(workspace, dev)
    if out is None:
        out = torch.empty((batch, s_next, h_q, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((batch, s_next, h_q), dtype=torch.float32, device=q.device)
    need = lib.sparse_mla_decode_workspace_size(batch, s_next, h_q, 512, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.sparse_mla_decode(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(cache_seqlens), _ptr(indices),
                               float(sm_scale), _ptr(out), _ptr(lse), batch, s_next, h_q, d_qk, 512, topk, page,
                               max_blocks, num_blocks, _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "sparse_mla_decode")
    return out, lse


FP8_SLOT_BYTES = 656


def sparse_mla_decode_fp8(q, kv_cache, block_table, cache_seqlens, indices, sm_scale, page_size=None,
                          workspace: Optional[torch.Tensor] = None, out=None, lse=None, stream=None):
    """Paged decode over an FP8 cache: kv_cache uint8 [num_blocks, page, 656]
    (512 e4m3 codes, 4 fp32 tile scales, 64 bf16 rope values per slot);
    everything else as sparse_mla_decode."""
    lib = load()
    batch, s_next, h_q, d_qk = q.shape
    num_blocks = kv_cache.shape[0]
    page = kv_cache.shape[1] if page_size is None else page_size
    max_blocks = block_table.shape[1]
    topk = indices.shape[-1]
    for t, dt, n in ((q, torch.bfloat16, "q"), (kv_cache, torch.uint8, "kv_cache"),
                     (block_table, torch.int32, "block_table"), (cache_seqlens, torch.int32, "cache_seqlens"),
                     (indices, torch.int32, "indices")):
        _need(t, dt, n)
    if kv_cache.shape[-1] != FP8_SLOT_BYTES:
        raise ValueError(f"kv_cache slots must be {FP8_SLOT_BYTES} bytes, got {kv_cache.shape[-1]}")
    dev = q.device
    _fits(kv_cache, num_blocks * page * FP8_SLOT_BYTES, "kv_cache", dev)
    _fits(block_table, batch * max_blocks, "block_table", dev)
    _fits(cache_seqlens, batch, "cache_seqlens", dev)
    _fits(indices, batch * s_next * topk, "indices", dev)
    _given(out, torch.bfloat16, "out", batch * s_next * h_q * 512, dev)
    _given(lse, torch.float32, "lse", batch * s_next * h_q, dev)
    _workspace(workspace, dev)
    if out is None:
        out = torch.empty((batch, s_next, h_q, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((batch, s_next, h_q), dtype=torch.float32, device=q.device)
    need = lib.sparse_mla_decode_workspace_size(batch, s_next, h_q, 512, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.sparse_mla_decode_fp8(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(cache_seqlens), _ptr(indices),
                                   float(sm_scale), _ptr(out), _ptr(lse), batch, s_next, h_q, d_qk, 512, topk, page,
                                   max_blocks, num_blocks, _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "sparse_mla_decode_fp8")
    return out, lse


# ---------------------------------------------------------------- debug: valid entries per token

def debug_valid_count(indices, s_kv: int, stream=None) -> torch.Tensor:
    """Valid entries of each token's list as the dense forward gathers them:
    indices [s_q, topk] int32 -> counts [s_q] int32."""
    lib = load()
    _need(indices, torch.int32, "indices")
    s_q, topk = indices.shape[0], indices.shape[-1]
    counts = torch.empty(s_q, dtype=torch.int32, device=indices.device)
    _check(lib.sparse_mla_debug_valid_count(_ptr(indices), s_q, int(s_kv), topk, _ptr(counts), _stream(stream)),
           "sparse_mla_debug_valid_count")
    return counts


def debug_valid_count_varlen(indices, cu_seqlens_q, cu_seqlens_kv, total_kv: int, stream=None) -> torch.Tensor:
    """As debug_valid_count for the packed layout of sparse_mla_fwd_varlen."""
    lib = load()
    for t, n in ((indices, "indices"), (cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_kv, "cu_seqlens_kv")):
        _need(t, torch.int32, n)
    total_q, topk = indices.shape[0], indices.shape[-1]
    batch = cu_seqlens_q.numel() - 1
    dev = indices.device
    _fits(cu_seqlens_q, batch + 1, "cu_seqlens_q", dev)
    _fits(cu_seqlens_kv, batch + 1, "cu_seqlens_kv", dev)
    counts = torch.empty(total_q, dtype=torch.int32, device=dev)
    _check(lib.sparse_mla_debug_valid_count_varlen(_ptr(indices), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), batch,
                                                   total_q, int(total_kv), topk, _ptr(counts), _stream(stream)),
           "sparse_mla_debug_valid_count_varlen")
    return counts


def debug_valid_count_paged(indices, block_table, cache_seqlens, page_size: int, num_blocks: int,
                            stream=None) -> torch.Tensor:
    """As debug_valid_count for the paged layout of sparse_mla_decode:
    indices [b, s_next, topk] -> counts [b * s_next] int32."""
    lib = load()
    for t, n in ((indices, "indices"), (block_table, "block_table"), (cache_seqlens, "cache_seqlens")):
        _need(t, torch.int32, n)
    batch, s_next, topk = indices.shape
    max_blocks = block_table.shape[1]
    dev = indices.device
    _fits(block_table, batch * max_blocks, "block_table", dev)
    _fits(cache_seqlens, batch, "cache_seqlens", dev)
    counts = torch.empty(batch * s_next, dtype=torch.int32, device=dev)
    _check(lib.sparse_mla_debug_valid_count_paged(_ptr(indices), _ptr(block_table), _ptr(cache_seqlens), batch,
                                                  s_next, topk, int(page_size), max_blocks, int(num_blocks),
                                                  _ptr(counts), _stream(stream)),
           "sparse_mla_debug_valid_count_paged")
    return counts


# ---------------------------------------------------------------- DSA indexer

def _seq_args(cu_seqlens_q, cu_seqlens_kv, device=None):
    if (cu_seqlens_q is None) != (cu_seqlens_kv is None):
        raise ValueError("give both cu_seqlens_q and cu_seqlens_kv, or neither")
    if cu_seqlens_q is None:
        return 1
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_kv, torch.int32, "cu_seqlens_kv")
    batch = cu_seqlens_q.numel() - 1
    if device is not None:
        _fits(cu_seqlens_q, batch + 1, "cu_seqlens_q", device)
        _fits(cu_seqlens_kv, batch + 1, "cu_seqlens_kv", device)
    return batch


def _workspace(workspace: Optional[torch.Tensor], device) -> None:
    if workspace is not None:
        _need(workspace, workspace.dtype, "workspace")
        _fits(workspace, 0, "workspace", device)


def _longest_kv(k_idx_rows: int, cu_seqlens_kv, max_seqlen_kv):
    if max_seqlen_kv is not None:
        return int(max_seqlen_kv)
    if cu_seqlens_kv is None:
        return int(k_idx_rows)
    if cu_seqlens_kv.numel() < 2:
        return 0
    return int((cu_seqlens_kv[1:] - cu_seqlens_kv[:-1]).max().item())   # a device read


def dsa_indexer_scores(q_idx, k_idx, weights, cu_seqlens_q=None, cu_seqlens_kv=None, row0: int = 0,
                       n_rows: Optional[int] = None, skip_len: int = 0, scores=None,
                       max_seqlen_kv: Optional[int] = None, stream=None):
    """Indexer scores of rows row0 .. row0+n_rows-1: q_idx [total_q,h_idx,128]
    bf16, k_idx [total_kv,128] bf16, weights [total_q,h_idx] fp32 ->
    scores [n_rows, row_stride] fp32 (row_stride = longest KV sequence
    rounded up to 4); positions a row does not see, and rows seeing at most
    skip_len positions, keep the given contents (-inf when allocated here)."""
    lib = load()
    total_q, h_idx, d_idx = q_idx.shape
    total_kv = k_idx.shape[0]
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_idx, torch.bfloat16, "k_idx")
    _need(weights, torch.float32, "weights")
    dev = q_idx.device
    _fits(k_idx, total_kv * d_idx, "k_idx", dev)
    _fits(weights, total_q * h_idx, "weights", dev)
    batch = _seq_args(cu_seqlens_q, cu_seqlens_kv, dev)
    n_rows = total_q - row0 if n_rows is None else n_rows
    stride = (_longest_kv(total_kv, cu_seqlens_kv, max_seqlen_kv) + 3) // 4 * 4
    if scores is None:
        scores = torch.full((n_rows, max(stride, 4)), float("-inf"), dtype=torch.float32, device=q_idx.device)
    else:
        _given(scores, torch.float32, "scores", max(n_rows, 0) * scores.shape[-1], dev)
    st = lib.dsa_indexer_scores(_ptr(q_idx), _ptr(k_idx), _ptr(weights), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
                                batch, total_q, total_kv, h_idx, d_idx, row0, n_rows, skip_len, _ptr(scores),
                                scores.shape[-1], _stream(stream))
    _check(st, "dsa_indexer_scores")
    return scores


def dsa_topk(scores, topk: int, total_q: int, total_kv: int, cu_seqlens_q=None, cu_seqlens_kv=None,
             row0: int = 0, n_rows: Optional[int] = None, indices=None, stream=None):
    """Lists of rows row0 .. row0+n_rows-1 from scores [n_rows, row_stride]
    fp32 -> indices [total_q, topk] int32 (only those rows written)."""
    lib = load()
    if scores is not None:
        _need(scores, torch.float32, "scores")
    n_rows = total_q - row0 if n_rows is None else n_rows
    dev = scores.device if scores is not None else (indices.device if indices is not None else torch.device("cuda"))
    batch = _seq_args(cu_seqlens_q, cu_seqlens_kv, dev)
    if scores is not None:
        _fits(scores, max(n_rows, 0) * scores.shape[-1], "scores", dev)
    if indices is None:
        indices = torch.full((total_q, topk), -2, dtype=torch.int32, device=dev)
    else:
        _given(indices, torch.int32, "indices", total_q * topk, dev)
    stride = scores.shape[-1] if scores is not None else 1
    st = lib.dsa_topk(_ptr(scores), stride, _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), batch, total_q, total_kv,
                      row0, n_rows, topk, _ptr(indices), _stream(stream))
    _check(st, "dsa_topk")
    return indices


def dsa_indexer_workspace_size(total_q: int, max_seqlen_kv: int, topk: int) -> int:
    return int(load().dsa_indexer_workspace_size(total_q, max_seqlen_kv, topk))


def dsa_indexer_topk(q_idx, k_idx, weights, topk: int, cu_seqlens_q=None, cu_seqlens_kv=None,
                     max_seqlen_kv: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                     indices=None, stream=None):
    """Index lists [total_q, topk] int32 of every query row (scores and
    top-k in query-row chunks sized by the workspace; a full-size workspace
    is allocated when none is given)."""
    lib = load()
    total_q, h_idx, d_idx = q_idx.shape
    total_kv = k_idx.shape[0]
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_idx, torch.bfloat16, "k_idx")
    _need(weights, torch.float32, "weights")
    dev = q_idx.device
    _fits(k_idx, total_kv * d_idx, "k_idx", dev)
    _fits(weights, total_q * h_idx, "weights", dev)
    batch = _seq_args(cu_seqlens_q, cu_seqlens_kv, dev)
    longest = _longest_kv(total_kv, cu_seqlens_kv, max_seqlen_kv)
    if indices is None:
        indices = torch.empty((total_q, topk), dtype=torch.int32, device=q_idx.device)
    else:
        _given(indices, torch.int32, "indices", total_q * topk, dev)
    _workspace(workspace, dev)
    if workspace is None:
        need = lib.dsa_indexer_workspace_size(total_q, longest, topk)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_idx.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.dsa_indexer_topk(_ptr(q_idx), _ptr(k_idx), _ptr(weights), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
                              batch, total_q, total_kv, longest, h_idx, d_idx, topk, _ptr(indices),
                              _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "dsa_indexer_topk")
    return indices


def _paged_args(q_idx, k_cache, weights, block_table, cache_seqlens):
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(weights, torch.float32, "weights")
    _need(block_table, torch.int32, "block_table")
    _need(cache_seqlens, torch.int32, "cache_seqlens")
    batch, s_next, h_idx, d_idx = q_idx.shape
    num_blocks, page = k_cache.shape[0], k_cache.shape[1]
    max_blocks = block_table.shape[1]
    dev = q_idx.device
    _fits(k_cache, num_blocks * page * d_idx, "k_cache", dev)
    _fits(weights, batch * s_next * h_idx, "weights", dev)
    _fits(block_table, batch * max_blocks, "block_table", dev)
    _fits(cache_seqlens, batch, "cache_seqlens", dev)
    return batch, s_next, h_idx, d_idx, page, max_blocks, num_blocks


def dsa_indexer_scores_paged(q_idx, k_cache, weights, block_table, cache_seqlens, max_seqlen_kv: int,
                             row0: int = 0, n_rows: Optional[int] = None, skip_len: int = 0, scores=None,
                             stream=None):
    """Decode indexer scores over a paged key cache: q_idx [b,s_next,h_idx,128],
    k_cache [num_blocks,64,128], weights [b,s_next,h_idx], block_table
    [b,max_blocks], cache_seqlens [b] -> scores [n_rows, row_stride] fp32 over
    the flattened rows b*s_next + j (-inf where not written)."""
    lib = load()
    batch, s_next, h_idx, d_idx, page, max_blocks, num_blocks = _paged_args(q_idx, k_cache, weights, block_table,
                                                                            cache_seqlens)
    n_rows = batch * s_next - row0 if n_rows is None else n_rows
    stride = (int(max_seqlen_kv) + 3) // 4 * 4
    if scores is None:
        scores = torch.full((n_rows, max(stride, 4)), float("-inf"), dtype=torch.float32, device=q_idx.device)
    else:
        _given(scores, torch.float32, "scores", max(n_rows, 0) * scores.shape[-1], q_idx.device)
    st = lib.dsa_indexer_scores_paged(_ptr(q_idx), _ptr(k_cache), _ptr(weights), _ptr(block_table),
                                      _ptr(cache_seqlens), batch, s_next, h_idx, d_idx, page, max_blocks, num_blocks,
                                      row0, n_rows, skip_len, _ptr(scores), scores.shape[-1], _stream(stream))
    _check(st, "dsa_indexer_scores_paged")
    return scores


def dsa_indexer_topk_paged(q_idx, k_cache, weights, block_table, cache_seqlens, topk: int,
                           max_seqlen_kv: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                           indices=None, stream=None):
    """Decode index lists [b, s_next, topk] int32 over a paged key cache
    (positions local to each request)."""
    lib = load()
    batch, s_next, h_idx, d_idx, page, max_blocks, num_blocks = _paged_args(q_idx, k_cache, weights, block_table,
                                                                            cache_seqlens)
    if max_seqlen_kv is None:
        max_seqlen_kv = int(cache_seqlens.max().item()) if cache_seqlens.numel() else 0   # a device read
    if indices is None:
        indices = torch.empty((batch, s_next, topk), dtype=torch.int32, device=q_idx.device)
    else:
        _given(indices, torch.int32, "indices", batch * s_next * topk, q_idx.device)
    _workspace(workspace, q_idx.device)
    if workspace is None:
        need = lib.dsa_indexer_workspace_size(batch * s_next, int(max_seqlen_kv), topk)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_idx.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.dsa_indexer_topk_paged(_ptr(q_idx), _ptr(k_cache), _ptr(weights), _ptr(block_table),
                                    _ptr(cache_seqlens), batch, s_next, h_idx, d_idx, page, max_blocks, num_blocks,
                                    int(max_seqlen_kv), topk, _ptr(indices), _ptr(workspace), ws_bytes,
                                    _stream(stream))
    _check(st, "dsa_indexer_topk_paged")
    return indices


def get_device_error() -> int:
    code = c_int(0)
    _check(load().sparse_mla_get_device_error(ctypes.byref(code)), "sparse_mla_get_device_error")
    return code.value


def clear_device_error():
    _check(load().sparse_mla_clear_device_error(), "sparse_mla_clear_device_error")


def set_wait_timeout_ns(ns: int):
    load().sparse_mla_set_wait_timeout_ns(int(ns))
