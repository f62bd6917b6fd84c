"""Python binding of the sparse-attention C ABI (include/nsa.h).

Argument marshalling only: every computation runs in libnsa.so's CUDA
kernels (the local virtual-batch builder runs in its host C++).  Device
buffers are torch CUDA tensors; work is enqueued on the current torch stream
unless `stream` is given.  There is no CPU fallback: if the library cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional

import numpy as np
import torch

from . import _build

__all__ = [
    "NsaError", "load", "MODE_DECODE", "MODE_EXTEND", "MODE_TARGET_VERIFY", "DT_F32", "DT_BF16",
    "DT_E4M3", "nsa_metadata", "alloc_metadata", "alloc_score_hist", "nsa_local_virtual_batches", "nsa_effective_chunk_size",
    "nsa_indexer_logits", "nsa_topk_transform", "nsa_topk_launches", "nsa_sparse_mla",
    "nsa_sparse_mla_workspace_bytes", "nsa_sparse_mla_plan", "nsa_set_mla_kv", "nsa_quantize_kv_cache", "nsa_dequantize_kv_paged",
    "nsa_set_index_k", "nsa_topk_transform_ragged", "nsa_flatten_page_table", "nsa_copy_buffers",
    "nsa_check_bounded_wait", "nsa_local_attention", "nsa_status_read", "nsa_status_string", "nsa_abi_version",
    "EXPORTED_SYMBOLS",
]

MODE_DECODE, MODE_EXTEND, MODE_TARGET_VERIFY = 0, 1, 2
DT_F32, DT_BF16, DT_E4M3 = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_BOUNDS, ERR_TIMEOUT = range(6)

EXPORTED_SYMBOLS = [
    "nsa_status_string", "nsa_abi_version", "nsa_status_read", "nsa_metadata",
    "nsa_effective_chunk_size", "nsa_local_virtual_batches", "nsa_indexer_logits",
    "nsa_topk_transform", "nsa_topk_workspace_bytes", "nsa_topk_launches", "nsa_sparse_mla",
    "nsa_sparse_mla_workspace_bytes",
    "nsa_sparse_mla_plan", "nsa_set_mla_kv", "nsa_quantize_kv_cache", "nsa_dequantize_kv_paged", "nsa_set_index_k",
    "nsa_topk_transform_ragged", "nsa_flatten_page_table", "nsa_copy_buffers",
    "nsa_check_bounded_wait", "nsa_local_attention",
]

_lib = None


class NsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {nsa_status_string(code)} ({code})")


def load(build_if_missing: bool = True):
    """Load libnsa.so (building it with nvcc when missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libnsa.so is missing ({path}); run __graft_entry__.build()")
    lib = C.CDLL(path)
    P, I, L, F, S = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_size_t
    sig = {
        "nsa_status_string": ([I], C.c_char_p),
        "nsa_abi_version": ([], I),
        "nsa_status_read": ([P, P, P], I),
        "nsa_metadata": ([I, I, I, I, I, I, I, P, P, P, L, L, P, P, P, P], I),
        "nsa_effective_chunk_size": ([I, I, I], I),
        "nsa_local_virtual_batches": ([I, I, I, P, P, P, L, L, I, P, P, P, P, P, P], I),
        "nsa_indexer_logits": ([I, P, P, P, P, L, I, I, I, P, L, P, P, I, I, I, P, L, P, P, P], I),
        "nsa_topk_transform": ([P, L, P, P, P, L, P, L, I, I, I, P, L, P, P, S, P, P], I),
        "nsa_topk_workspace_bytes": ([I, I, I], S),
        "nsa_topk_launches": ([I, I, I], I),
        "nsa_sparse_mla": ([I, I, P, L, L, P, L, L, P, L, P, L, I, I, I, I, I, F, P, P, P, S, P, P], I),
        "nsa_sparse_mla_workspace_bytes": ([I, I, I, I, I, I, I], S),
        "nsa_sparse_mla_plan": ([I, I, I, I, I, I, I, P, P], I),
        "nsa_set_mla_kv": ([I, P, L, P, L, P, I, I, I, P, L, P, P], I),
        "nsa_quantize_kv_cache": ([P, L, I, I, P, P], I),
        "nsa_dequantize_kv_paged": ([P, L, I, I, P, L, P, P, P], I),
        "nsa_set_index_k": ([P, L, P, I, I, P, P, L, P, P], I),
        "nsa_topk_transform_ragged": ([P, L, P, P, P, I, I, I, P, L, P, P, S, P, P], I),
        "nsa_flatten_page_table": ([I, P, L, P, P, P, L, P, P], I),
        "nsa_copy_buffers": ([I, P, P, P, P], I),
        "nsa_check_bounded_wait": ([P, C.c_longlong, P], I),
        "nsa_local_attention": ([P, L, P, P, L, I, P, L, P, P, I, I, I, I, I, F, P, P, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    _lib = lib
    return lib


class _MetadataOut(C.Structure):
    _fields_ = [("cache_seqlens", C.c_void_p), ("cu_seqlens_k", C.c_void_p), ("cu_seqlens_q", C.c_void_p),
                ("seqlens_expanded", C.c_void_p), ("nsa_cache_seqlens", C.c_void_p),
                ("nsa_cu_seqlens_k", C.c_void_p), ("nsa_cu_seqlens_q", C.c_void_p),
                ("row_to_req", C.c_void_p), ("page_table_1", C.c_void_p), ("page_table_1_ld", C.c_int64),
                ("real_page_table", C.c_void_p), ("real_page_table_ld", C.c_int64),
                ("indexer_ks", C.c_void_p), ("indexer_ke", C.c_void_p), ("req_rows", C.c_void_p)]


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _ld(t: torch.Tensor) -> int:
    """Leading dimension of a row-major 2D tensor: its row stride, or for a single
    row (whose stride is arbitrary, 0 for a broadcast view) its row length.  The
    library reads every row as packed, so elements of a row must be adjacent."""
    if t.dim() != 2:
        raise ValueError(f"expected a 2D tensor, got shape {tuple(t.shape)}")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("the elements of each row must be adjacent (stride 1 in the last dimension)")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def alloc_score_hist(R: int, device="cuda") -> torch.Tensor:
    """A zeroed [R, 2048] uint32 (stored as int32) digit-count buffer shared by
    nsa_indexer_logits and nsa_topk_transform (the top-k leaves it zeroed)."""
    return torch.zeros((max(R, 1), 2048), dtype=torch.int32, device=device)


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, code: int):
    if code != OK:
        raise NsaError(fn, code)


def nsa_status_string(code: int) -> str:
    return load().nsa_status_string(code).decode()


def nsa_abi_version() -> int:
    return load().nsa_abi_version()


def nsa_status_read(status: torch.Tensor, stream=None) -> int:
    """Synchronize `stream` and return the device status word."""
    v = C.c_int32(0)
    _check("nsa_status_read", load().nsa_status_read(_ptr(status), C.byref(v), _stream(stream)))
    return int(v.value)


# ------------------------------------------------------------------ metadata

def alloc_metadata(mode: int, B: int, R: int, W: int, page_size: int, device="cuda",
                   with_ks_ke: bool = False, with_page_table_1: bool = True,
                   with_req_rows: bool = False) -> Dict[str, torch.Tensor]:
    """Device buffers for nsa_metadata's outputs (page_table_1 left out, and so not
    written, when with_page_table_1 is False; req_rows added with with_req_rows)."""
    i32 = dict(dtype=torch.int32, device=device)
    nq = R + 1 if mode == MODE_TARGET_VERIFY else B + 1
    npg = (W + page_size - 1) // page_size
    out = dict(cache_seqlens=torch.empty(B, **i32), cu_seqlens_k=torch.empty(B + 1, **i32),
               cu_seqlens_q=torch.empty(nq, **i32), seqlens_expanded=torch.empty(R, **i32),
               nsa_cache_seqlens=torch.empty(R, **i32), nsa_cu_seqlens_k=torch.empty(R + 1, **i32),
               nsa_cu_seqlens_q=torch.empty(R + 1, **i32), row_to_req=torch.empty(R, **i32),
               real_page_table=torch.empty((B, max(npg, 1)), **i32))
    if with_page_table_1:
        out["page_table_1"] = torch.empty((B, max(W, 1)), **i32)
    if with_req_rows:
        out["req_rows"] = torch.empty(B, **i32)
    if with_ks_ke:
        out["indexer_ks"] = torch.empty(R, **i32)
        out["indexer_ke"] = torch.empty(R, **i32)
    return out


def nsa_metadata(mode: int, B: int, R: int, W: int, n_draft: int, topk: int, page_size: int,
                 seq_lens: torch.Tensor, extend_lens: Optional[torch.Tensor], req_to_token: torch.Tensor,
                 req_pool_indices: torch.Tensor, out: Dict[str, torch.Tensor],
                 status: Optional[torch.Tensor] = None, stream=None) -> None:
    pt1 = out.get("page_table_1")
    o = _MetadataOut(*(_ptr(out[k]) for k in ["cache_seqlens", "cu_seqlens_k", "cu_seqlens_q",
                                              "seqlens_expanded", "nsa_cache_seqlens", "nsa_cu_seqlens_k",
                                              "nsa_cu_seqlens_q", "row_to_req"]),
                     _ptr(pt1), _ld(pt1) if pt1 is not None else 0, _ptr(out["real_page_table"]),
                     _ld(out["real_page_table"]), _ptr(out.get("indexer_ks")), _ptr(out.get("indexer_ke")),
                     _ptr(out.get("req_rows")))
    rc = load().nsa_metadata(mode, B, R, W, n_draft, topk, page_size, _ptr(seq_lens), _ptr(extend_lens),
                             _ptr(req_to_token), _ld(req_to_token), req_to_token.shape[0],
                             _ptr(req_pool_indices), C.byref(o), _ptr(status), _stream(stream))
    _check("nsa_metadata", rc)


# ------------------------------------------------------------------ local attention (host)

def nsa_effective_chunk_size(attn_chunk_size: int, max_seq_len: int, page_size: int) -> int:
    v = load().nsa_effective_chunk_size(attn_chunk_size, max_seq_len, page_size)
    if v < 0:
        raise NsaError("nsa_effective_chunk_size", ERR_INVALID_ARG)
    return v


def nsa_local_virtual_batches(attn_chunk_size: int, page_size: int, cu_seqlens_q, seq_lens, block_table):
    """Host call.  Returns numpy arrays (seqlens_q_local, cu_seqlens_q_local,
    seqlens_k_local, k_seqstarts_absolute, block_table_local)."""
    lib = load()
    cq = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    B = len(sl)
    n = C.c_int(0)
    P = lambda a: a.ctypes.data_as(C.c_void_p)
    _check("nsa_local_virtual_batches",
           lib.nsa_local_virtual_batches(attn_chunk_size, page_size, B, P(cq), P(sl), P(bt), bt.shape[1],
                                         bt.shape[1], 0, C.byref(n), None, None, None, None, None))
    V, ppl = n.value, attn_chunk_size // page_size
    sq, cu, sk = np.zeros(V, np.int32), np.zeros(V + 1, np.int32), np.zeros(V, np.int32)
    st, btl = np.zeros(V, np.int32), np.zeros((V, ppl), np.int32)
    _check("nsa_local_virtual_batches",
           lib.nsa_local_virtual_batches(attn_chunk_size, page_size, B, P(cq), P(sl), P(bt), bt.shape[1],
                                         bt.shape[1], V, C.byref(n), P(sq), P(cu), P(sk), P(st), P(btl)))
    return sq, cu, sk, st, btl


# ------------------------------------------------------------------ indexer / top-k / attention

def nsa_indexer_logits(dtype: int, q_idx: torch.Tensor, weights: torch.Tensor, k_cache: torch.Tensor,
                       k_scale: torch.Tensor, real_page_table: torch.Tensor, row_to_req: torch.Tensor,
                       row_len: torch.Tensor, max_row_len: int, logits: torch.Tensor,
                       status: Optional[torch.Tensor] = None, stream=None, rows_per_group: int = 1,
                       score_hist: Optional[torch.Tensor] = None) -> None:
    R, Hi, Di = q_idx.shape
    num_pages, ps = k_cache.shape[0], k_cache.shape[1]
    assert q_idx.is_contiguous() and k_cache.is_contiguous() and weights.is_contiguous() and k_scale.is_contiguous()
    rc = load().nsa_indexer_logits(dtype, _ptr(q_idx), _ptr(weights), _ptr(k_cache), _ptr(k_scale), num_pages,
                                   ps, Hi, Di, _ptr(real_page_table), _ld(real_page_table),
                                   _ptr(row_to_req), _ptr(row_len), R, rows_per_group, max_row_len, _ptr(logits),
                                   _ld(logits), _ptr(_hist(score_hist, R)), _ptr(status), _stream(stream))
    _check("nsa_indexer_logits", rc)


def _hist(h: Optional[torch.Tensor], R: int) -> Optional[torch.Tensor]:
    if h is not None:
        assert h.is_contiguous() and h.element_size() == 4 and h.shape[-1] == 2048 and h.numel() >= R * 2048
    return h


def nsa_topk_workspace_bytes(R: int, max_row_len: int, with_score_hist: bool) -> int:
    return int(load().nsa_topk_workspace_bytes(R, max_row_len, 1 if with_score_hist else 0))


def nsa_topk_launches(R: int, max_row_len: int, with_score_hist: bool) -> int:
    return int(load().nsa_topk_launches(R, max_row_len, 1 if with_score_hist else 0))


def alloc_topk_workspace(R: int, max_row_len: int, with_score_hist: bool, device="cuda") -> torch.Tensor:
    """A zeroed top-k workspace (the calls leave it zeroed for the next one)."""
    n = max(256, nsa_topk_workspace_bytes(R, max_row_len, with_score_hist))
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _topk_ws(ws: Optional[torch.Tensor], R: int, max_row_len: int, score_hist, device):
    if ws is None:  # a fresh zeroed one (a caller running many steps keeps its own)
        ws = alloc_topk_workspace(R, max_row_len, score_hist is not None, device)
    return ws, ws.numel() * ws.element_size()


def nsa_topk_transform(logits: torch.Tensor, row_len: torch.Tensor, row_to_req: torch.Tensor,
                       page_table_1: torch.Tensor, topk: int, max_row_len: int, indices: torch.Tensor,
                       status: Optional[torch.Tensor] = None, stream=None,
                       score_hist: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       pt_rows: Optional[torch.Tensor] = None) -> None:
    """pt_rows: request b's slots are row pt_rows[b] of page_table_1 (e.g. req_to_token
    with nsa_metadata's req_rows); None: row b."""
    R = row_len.shape[0]
    ws, ws_bytes = _topk_ws(workspace, R, max_row_len, score_hist, logits.device)
    rc = load().nsa_topk_transform(_ptr(logits), _ld(logits), _ptr(row_len), _ptr(row_to_req),
                                   _ptr(page_table_1), _ld(page_table_1), _ptr(pt_rows),
                                   int(page_table_1.shape[0]) if pt_rows is not None else 0, R, topk, max_row_len,
                                   _ptr(indices), _ld(indices), _ptr(_hist(score_hist, R)), _ptr(ws), ws_bytes,
                                   _ptr(status), _stream(stream))
    _check("nsa_topk_transform", rc)


def nsa_sparse_mla_workspace_bytes(q_dtype: int, kv_dtype: int, R: int, H: int, d_latent: int, d_rope: int,
                                   topk: int) -> int:
    return int(load().nsa_sparse_mla_workspace_bytes(q_dtype, kv_dtype, R, H, d_latent, d_rope, topk))


def nsa_sparse_mla_plan(q_dtype: int, kv_dtype: int, R: int, H: int, d_latent: int, d_rope: int,
                        topk: int):
    """(splits per top-k list, kernel launches per call) of nsa_sparse_mla for this shape."""
    ns, nl = C.c_int(0), C.c_int(0)
    _check("nsa_sparse_mla_plan", load().nsa_sparse_mla_plan(q_dtype, kv_dtype, R, H, d_latent, d_rope, topk,
                                                             C.byref(ns), C.byref(nl)))
    return int(ns.value), int(nl.value)


def nsa_sparse_mla(q_dtype: int, kv_dtype: int, q_nope: torch.Tensor, q_rope: torch.Tensor, kv: torch.Tensor,
                   indices: torch.Tensor, sm_scale: float, out: torch.Tensor, lse: torch.Tensor,
                   workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                   stream=None, num_slots: Optional[int] = None) -> None:
    """q_nope [R,H,d_latent] and q_rope [R,H,d_rope] (any row / head strides,
    unit stride in the last dim); kv [slots, row]; indices [R, topk]."""
    R, H, d_latent = q_nope.shape
    d_rope = q_rope.shape[2]
    topk = indices.shape[1]
    assert q_nope.stride(2) == 1 and q_rope.stride(2) == 1 and out.is_contiguous() and lse.is_contiguous()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().nsa_sparse_mla(q_dtype, kv_dtype, _ptr(q_nope), q_nope.stride(0), q_nope.stride(1), _ptr(q_rope),
                               q_rope.stride(0), q_rope.stride(1), _ptr(kv),
                               kv.shape[0] if num_slots is None else num_slots, _ptr(indices),
                               _ld(indices), R, H, d_latent, d_rope, topk, float(sm_scale), _ptr(out),
                               _ptr(lse), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream))
    _check("nsa_sparse_mla", rc)


# ---------------------------------------------------------------- KV-cache write side

def nsa_set_mla_kv(kv_dtype: int, k_nope: torch.Tensor, k_rope: torch.Tensor, loc: torch.Tensor,
                   kv: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """New tokens' latent [n, 512] and rope [n, 64] (bf16) into the KV cache at slots `loc` (int32)."""
    n = loc.shape[0]
    num_slots = kv.shape[0]
    rc = load().nsa_set_mla_kv(kv_dtype, _ptr(k_nope), k_nope.stride(0), _ptr(k_rope), k_rope.stride(0), _ptr(loc),
                               n, k_nope.shape[1], k_rope.shape[1], _ptr(kv), num_slots, _ptr(status),
                               _stream(stream))
    _check("nsa_set_mla_kv", rc)


def nsa_quantize_kv_cache(kv_bf16: torch.Tensor, kv_fp8: torch.Tensor, d_latent: int = 512, d_rope: int = 64,
                          stream=None) -> None:
    rc = load().nsa_quantize_kv_cache(_ptr(kv_bf16), kv_bf16.shape[0], d_latent, d_rope, _ptr(kv_fp8),
                                      _stream(stream))
    _check("nsa_quantize_kv_cache", rc)


def nsa_dequantize_kv_paged(kv_fp8: torch.Tensor, slots: torch.Tensor, out_bf16: torch.Tensor,
                            d_latent: int = 512, d_rope: int = 64, status: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    rc = load().nsa_dequantize_kv_paged(_ptr(kv_fp8), kv_fp8.shape[0], d_latent, d_rope, _ptr(slots),
                                        slots.shape[0], _ptr(out_bf16), _ptr(status), _stream(stream))
    _check("nsa_dequantize_kv_paged", rc)


def nsa_set_index_k(k: torch.Tensor, loc: torch.Tensor, k_cache: torch.Tensor, k_scale: torch.Tensor,
                    status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Indexer keys [n, 128] (bf16) -> e4m3 codes and fp32 scales at slots `loc` of the paged key cache."""
    num_slots = k_scale.numel()
    rc = load().nsa_set_index_k(_ptr(k), k.stride(0), _ptr(loc), loc.shape[0], k.shape[1], _ptr(k_cache),
                                _ptr(k_scale), num_slots, _ptr(status), _stream(stream))
    _check("nsa_set_index_k", rc)


# ---------------------------------------------------------------- RAGGED extend

def nsa_topk_transform_ragged(logits: torch.Tensor, row_len: torch.Tensor, row_to_req: torch.Tensor,
                              req_offset: torch.Tensor, topk: int, max_row_len: int, indices: torch.Tensor,
                              status: Optional[torch.Tensor] = None, stream=None,
                              score_hist: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None) -> None:
    R = row_len.shape[0]
    ws, ws_bytes = _topk_ws(workspace, R, max_row_len, score_hist, logits.device)
    rc = load().nsa_topk_transform_ragged(_ptr(logits), _ld(logits), _ptr(row_len), _ptr(row_to_req),
                                          _ptr(req_offset), R, topk, max_row_len, _ptr(indices), _ld(indices),
                                          _ptr(_hist(score_hist, R)), _ptr(ws), ws_bytes, _ptr(status),
                                          _stream(stream))
    _check("nsa_topk_transform_ragged", rc)


def nsa_flatten_page_table(page_table_1: torch.Tensor, kv_len: torch.Tensor, kv_start: torch.Tensor,
                           out: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    B = kv_len.shape[0]
    rc = load().nsa_flatten_page_table(B, _ptr(page_table_1), _ld(page_table_1), _ptr(kv_len), _ptr(kv_start),
                                       _ptr(out), out.numel(), _ptr(status), _stream(stream))
    _check("nsa_flatten_page_table", rc)


# ---------------------------------------------------------------- copies

def nsa_copy_buffers(pairs, stream=None) -> None:
    """[(dst, src), ...] tensors of equal byte size (device or pinned host), copied in one launch."""
    n = len(pairs)
    src = (C.c_void_p * max(1, n))(*[p[1].data_ptr() for p in pairs])
    dst = (C.c_void_p * max(1, n))(*[p[0].data_ptr() for p in pairs])
    nb = (C.c_int64 * max(1, n))(*[p[1].numel() * p[1].element_size() for p in pairs])
    for d, s in pairs:
        assert d.numel() * d.element_size() == s.numel() * s.element_size()
    _check("nsa_copy_buffers", load().nsa_copy_buffers(n, src, dst, nb, _stream(stream)))


def nsa_check_bounded_wait(status: torch.Tensor, budget_cycles: int, stream=None) -> None:
    _check("nsa_check_bounded_wait", load().nsa_check_bounded_wait(_ptr(status), int(budget_cycles), _stream(stream)))


# ---------------------------------------------------------------- chunk-local attention

def nsa_local_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                        cu_seqlens_q: torch.Tensor, seqused_k: torch.Tensor, sm_scale: float, out: torch.Tensor,
                        lse: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q bf16 [total_q, Hq, D] (rows may be strided); k_cache / v_cache bf16 [pages, page_size, Hkv, D];
    block_table int32 [nvb, bt_ld]; cu_seqlens_q int32 [nvb + 1]; seqused_k int32 [nvb];
    out bf16 [total_q, Hq, D]; lse float32 [total_q, Hq]."""
    total_q, Hq, D = q.shape
    assert q.stride(2) == 1 and q.stride(1) == D
    num_pages, ps, Hkv, Dk = k_cache.shape
    assert Dk == D and tuple(v_cache.shape) == tuple(k_cache.shape)
    assert k_cache.is_contiguous() and v_cache.is_contiguous() and block_table.stride(1) == 1
    assert out.is_contiguous() and lse.is_contiguous()
    nvb = seqused_k.shape[0]
    # the library reads bt_ld as the row stride and as the row's capacity: a column
    # slice of a wider table (stride beyond the row length) would overstate it
    if block_table.shape[0] > 1 and block_table.stride(0) != block_table.shape[1]:
        raise ValueError("block_table rows must be packed (row stride == row length)")
    bt_ld = _ld(block_table)
    rc = load().nsa_local_attention(_ptr(q), q.stride(0), _ptr(k_cache), _ptr(v_cache), num_pages, ps,
                                    _ptr(block_table), bt_ld, _ptr(cu_seqlens_q), _ptr(seqused_k),
                                    nvb, total_q, Hq, Hkv, D, float(sm_scale), _ptr(out), _ptr(lse), _ptr(status),
                                    _stream(stream))
    _check("nsa_local_attention", rc)
