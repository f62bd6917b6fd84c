"""The oracle: TEST INFRASTRUCTURE, not part of the product.

A ctypes front end to `nsa_oracle.c`, a plain single-threaded C99 statement of
the sparse-attention path in double precision.  Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import this package; the product
library never does, and the two share no code.

`build()` compiles the C file with gcc (no fast-math, no FMA contraction) into
`oracle/_build/liboracle.so` on first use.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nsa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_DECODE, MODE_EXTEND, MODE_VERIFY = 0, 1, 2
DT_F32, DT_BF16, DT_E4M3 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _library_path() -> str:
    """The compiled oracle to load: `NSA_ORACLE_LIB` names a prebuilt copy (the
    mutation tests load builds with a planted mistake this way), else `build()`."""
    alt = os.environ.get("NSA_ORACLE_LIB")
    return alt if alt else build()


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(_library_path())
            P, I, L, D = C.c_void_p, C.c_int, C.c_int64, C.c_double
            lib.orc_e4m3_to_f64.argtypes, lib.orc_e4m3_to_f64.restype = [C.c_uint8], D
            lib.orc_bf16_to_f64.argtypes, lib.orc_bf16_to_f64.restype = [C.c_uint16], D
            lib.orc_num_rows.argtypes, lib.orc_num_rows.restype = [I, I, P, I], L
            lib.orc_metadata.argtypes = [I, I, I, I, I, I, P, P, P, L, P] + [P] * 8 + [P, L, P, L, P, P]
            lib.orc_metadata.restype = L
            lib.orc_effective_chunk_size.argtypes, lib.orc_effective_chunk_size.restype = [I, I, I], I
            lib.orc_local_virtual_batches.argtypes = [I, I, I, P, P, P, L, I, P, P, P, P, P]
            lib.orc_local_virtual_batches.restype = I
            lib.orc_indexer_row.argtypes = [I, I, I, I, L, P, P, P, P, P, I, P]
            lib.orc_indexer_row.restype = I
            lib.orc_topk_row.argtypes, lib.orc_topk_row.restype = [P, I, I, P, P], I
            lib.orc_fp8_row_bytes.argtypes, lib.orc_fp8_row_bytes.restype = [I, I], L
            lib.orc_sparse_mla_row.argtypes = [I, I, I, I, I, I, P, L, P, L, P, L, P, D, P, P]
            lib.orc_sparse_mla_row.restype = I
            lib.orc_e4m3_encode.argtypes, lib.orc_e4m3_encode.restype = [C.c_float], C.c_uint8
            lib.orc_f32_to_bf16.argtypes, lib.orc_f32_to_bf16.restype = [C.c_float], C.c_uint16
            lib.orc_quantize_mla_row.argtypes, lib.orc_quantize_mla_row.restype = [P, P, I, I, P], None
            lib.orc_dequantize_mla_row.argtypes, lib.orc_dequantize_mla_row.restype = [P, I, I, P], None
            lib.orc_quantize_index_row.argtypes, lib.orc_quantize_index_row.restype = [P, I, P], C.c_float
            lib.orc_topk_ragged_row.argtypes, lib.orc_topk_ragged_row.restype = [P, I, I, C.c_int32, P], I
            lib.orc_flatten_page_table.argtypes, lib.orc_flatten_page_table.restype = [I, P, L, P, P], L
            lib.orc_local_attention_row.argtypes = [I, I, I, I, I, I, L, P, L, P, P, P, P, P, D, P, P]
            lib.orc_local_attention_row.restype = I
            _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats

def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    table = np.array([lib.orc_e4m3_to_f64(i) for i in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    flat = np.array([lib.orc_bf16_to_f64(int(x)) for x in b.reshape(-1)], dtype=np.float64)
    return flat.reshape(b.shape)


def fp8_row_bytes(d_latent: int, d_rope: int) -> int:
    return int(_load().orc_fp8_row_bytes(d_latent, d_rope))


# ---------------------------------------------------------------- metadata

def num_rows(mode: int, B: int, extend_lens=None, n_draft: int = 0) -> int:
    ext = None if extend_lens is None else _c(extend_lens, np.int32)
    return int(_load().orc_num_rows(mode, B, _p(ext), n_draft))


def metadata(mode: int, seq_lens, req_to_token, req_pool_indices, *, W: int, topk: int,
             page_size: int, extend_lens=None, n_draft: int = 0) -> dict:
    """All per-step metadata arrays (see orc_metadata)."""
    lib = _load()
    sl = _c(seq_lens, np.int32)
    B = len(sl)
    ext = None if extend_lens is None else _c(extend_lens, np.int32)
    r2t = _c(req_to_token, np.int32)
    rpi = _c(req_pool_indices, np.int32)
    R = num_rows(mode, B, ext, n_draft)
    nq = R + 1 if mode == MODE_VERIFY else B + 1
    npg = (W + page_size - 1) // page_size
    o = dict(cache_seqlens=np.zeros(B, np.int32), cu_seqlens_k=np.zeros(B + 1, np.int32),
             cu_seqlens_q=np.zeros(nq, np.int32), seqlens_expanded=np.zeros(R, np.int32),
             nsa_cache_seqlens=np.zeros(R, np.int32), nsa_cu_seqlens_k=np.zeros(R + 1, np.int32),
             nsa_cu_seqlens_q=np.zeros(R + 1, np.int32), row_to_req=np.zeros(R, np.int32),
             page_table_1=np.zeros((B, max(W, 1)), np.int32),
             real_page_table=np.zeros((B, max(npg, 1)), np.int32))
    if mode == MODE_EXTEND:
        o["indexer_ks"] = np.zeros(R, np.int32)
        o["indexer_ke"] = np.zeros(R, np.int32)
    ret = lib.orc_metadata(mode, B, W, n_draft, topk, page_size, _p(sl), _p(ext), _p(r2t),
                           r2t.shape[1], _p(rpi), _p(o["cache_seqlens"]), _p(o["cu_seqlens_k"]),
                           _p(o["cu_seqlens_q"]), _p(o["seqlens_expanded"]),
                           _p(o["nsa_cache_seqlens"]), _p(o["nsa_cu_seqlens_k"]),
                           _p(o["nsa_cu_seqlens_q"]), _p(o["row_to_req"]), _p(o["page_table_1"]),
                           o["page_table_1"].shape[1], _p(o["real_page_table"]),
                           o["real_page_table"].shape[1], _p(o.get("indexer_ks")),
                           _p(o.get("indexer_ke")))
    if ret < 0:
        raise ValueError(f"oracle metadata rejected its input ({ret})")
    o["page_table_1"] = o["page_table_1"][:, :W]
    o["real_page_table"] = o["real_page_table"][:, :npg]
    o["R"] = R
    return o


def effective_chunk_size(chunk: int, max_seq_len: int, page_size: int) -> int:
    return int(_load().orc_effective_chunk_size(chunk, max_seq_len, page_size))


def local_virtual_batches(chunk: int, page_size: int, cu_seqlens_q, seq_lens, block_table):
    """(seqlens_q_local, cu_seqlens_q_local, seqlens_k_local, k_seqstarts_absolute,
    block_table_local)"""
    lib = _load()
    cq = _c(cu_seqlens_q, np.int32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_table, np.int32)
    B = len(sl)
    n = lib.orc_local_virtual_batches(chunk, page_size, B, _p(cq), _p(sl), _p(bt), bt.shape[1],
                                      0, None, None, None, None, None)
    if n < 0:
        raise ValueError("oracle rejected the local-attention arguments")
    ppl = chunk // page_size
    sq, cu = np.zeros(n, np.int32), np.zeros(n + 1, np.int32)
    sk, st = np.zeros(n, np.int32), np.zeros(n, np.int32)
    btl = np.zeros((n, ppl), np.int32)
    m = lib.orc_local_virtual_batches(chunk, page_size, B, _p(cq), _p(sl), _p(bt), bt.shape[1], n,
                                      _p(sq), _p(cu), _p(sk), _p(st), _p(btl))
    assert m == n
    return sq, cu, sk, st, btl


# ---------------------------------------------------------------- indexer

def indexer_logits(dtype: int, q_idx, weights, k_cache, k_scale, real_page_table, row_to_req,
                   row_len, rows: Optional[Sequence[int]] = None, width: Optional[int] = None):
    """Logits for the given rows (all rows by default).

    Returns float32 [len(rows), width]; entries at s >= row_len are NaN.
    """
    lib = _load()
    q = np.ascontiguousarray(q_idx)
    w = _c(weights, np.float32)
    kc = np.ascontiguousarray(k_cache)
    ks = _c(k_scale, np.float32)
    rpt = _c(real_page_table, np.int32)
    r2q = _c(row_to_req, np.int32)
    rl = _c(row_len, np.int32)
    R, Hi, Di = q.shape
    num_pages, ps = kc.shape[0], kc.shape[1]
    rows = list(range(R)) if rows is None else list(rows)
    width = int(rl.max()) if width is None else width
    out = np.full((len(rows), max(width, 1)), np.nan, dtype=np.float32)
    esz = q.dtype.itemsize
    for i, r in enumerate(rows):
        L = int(rl[r])
        qp = C.c_void_p(q.ctypes.data + r * Hi * Di * esz)
        wp = C.c_void_p(w.ctypes.data + r * Hi * 4)
        tp = C.c_void_p(rpt.ctypes.data + int(r2q[r]) * rpt.shape[1] * 4)
        op = C.c_void_p(out.ctypes.data + i * out.shape[1] * 4)
        rc = lib.orc_indexer_row(dtype, Hi, Di, ps, num_pages, qp, wp, _p(kc), _p(ks), tp, L, op)
        if rc != 0:
            raise ValueError(f"oracle indexer: page id out of range in row {r}")
    return out[:, :width]


# ---------------------------------------------------------------- top-k

def topk_transform(logits, row_len, row_to_req, page_table_1, topk: int,
                   rows: Optional[Sequence[int]] = None, logits_rows_are_subset: bool = False):
    """indices int32 [len(rows), topk]: KV slots of each row's top-k (ascending
    token position), padded with -1.  `logits` holds one row per requested row
    when `logits_rows_are_subset`, else one row per query row."""
    lib = _load()
    lg = _c(logits, np.float32)
    rl = _c(row_len, np.int32)
    r2q = _c(row_to_req, np.int32)
    pt = _c(page_table_1, np.int32)
    rows = list(range(len(rl))) if rows is None else list(rows)
    out = np.zeros((len(rows), topk), dtype=np.int32)
    for i, r in enumerate(rows):
        lrow = i if logits_rows_are_subset else r
        L = int(rl[r])
        if L > lg.shape[1]:
            raise ValueError("row length exceeds the logits width")
        lp = C.c_void_p(lg.ctypes.data + lrow * lg.shape[1] * 4)
        tp = C.c_void_p(pt.ctypes.data + int(r2q[r]) * pt.shape[1] * 4)
        op = C.c_void_p(out.ctypes.data + i * topk * 4)
        lib.orc_topk_row(lp, L, topk, tp, op)
    return out


# ---------------------------------------------------------------- sparse MLA

def sparse_mla(q_dtype: int, kv_dtype: int, q_nope, q_rope, kv, indices, sm_scale: float,
               rows: Optional[Sequence[int]] = None, indices_rows_are_subset: bool = False):
    """(out float64 [n, H, d_latent], lse float64 [n, H]) for the given rows."""
    lib = _load()
    qn = np.ascontiguousarray(q_nope)
    qr = np.ascontiguousarray(q_rope)
    kvc = np.ascontiguousarray(kv)
    idx = _c(indices, np.int32)
    R, H, d_latent = qn.shape
    d_rope = qr.shape[2]
    topk = idx.shape[1]
    if kv_dtype == DT_E4M3:
        num_slots = kvc.shape[0]
        assert kvc.shape[1] == fp8_row_bytes(d_latent, d_rope)
    else:
        num_slots = kvc.shape[0]
    rows = list(range(R)) if rows is None else list(rows)
    out = np.zeros((len(rows), H, d_latent), dtype=np.float64)
    lse = np.zeros((len(rows), H), dtype=np.float64)
    esz = qn.dtype.itemsize
    for i, r in enumerate(rows):
        irow = i if indices_rows_are_subset else r
        qn_p = C.c_void_p(qn.ctypes.data + r * H * d_latent * esz)
        qr_p = C.c_void_p(qr.ctypes.data + r * H * d_rope * esz)
        ip = C.c_void_p(idx.ctypes.data + irow * topk * 4)
        op = C.c_void_p(out.ctypes.data + i * H * d_latent * 8)
        lp = C.c_void_p(lse.ctypes.data + i * H * 8)
        rc = lib.orc_sparse_mla_row(q_dtype, kv_dtype, H, d_latent, d_rope, topk, qn_p, d_latent,
                                    qr_p, d_rope, _p(kvc), num_slots, ip, float(sm_scale), op, lp)
        if rc != 0:
            raise ValueError(f"oracle sparse MLA: index out of range in row {r}")
    return out, lse


# ---------------------------------------------------------------- KV-cache write side

def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> e4m3 codes (nearest, ties to even, saturating at 448)."""
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.orc_e4m3_encode(float(v)) for v in a.reshape(-1)], dtype=np.uint8).reshape(a.shape)


def f32_to_bf16(x) -> np.ndarray:
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in a.reshape(-1)], dtype=np.uint16).reshape(a.shape)


def quantize_mla_rows(latent, rope) -> np.ndarray:
    """bf16 bits [N, d_latent] and [N, d_rope] -> fp8 rows uint8 [N, row_bytes]."""
    lib = _load()
    lat = _c(latent, np.uint16)
    rp = _c(rope, np.uint16)
    n, dl = lat.shape
    dr = rp.shape[1]
    out = np.zeros((n, fp8_row_bytes(dl, dr)), dtype=np.uint8)
    for i in range(n):
        lib.orc_quantize_mla_row(_p(lat[i]), _p(rp[i]), dl, dr, _p(out[i]))
    return out


def dequantize_mla_rows(rows, d_latent: int, d_rope: int) -> np.ndarray:
    """fp8 rows uint8 [N, row_bytes] -> bf16 bits [N, d_latent + d_rope]."""
    lib = _load()
    r = _c(rows, np.uint8)
    out = np.zeros((r.shape[0], d_latent + d_rope), dtype=np.uint16)
    for i in range(r.shape[0]):
        lib.orc_dequantize_mla_row(_p(r[i]), d_latent, d_rope, _p(out[i]))
    return out


def quantize_index_rows(k):
    """bf16 bits [N, D] -> (e4m3 codes [N, D], fp32 scales [N])."""
    lib = _load()
    a = _c(k, np.uint16)
    codes = np.zeros(a.shape, dtype=np.uint8)
    scales = np.zeros((a.shape[0],), dtype=np.float32)
    for i in range(a.shape[0]):
        scales[i] = lib.orc_quantize_index_row(_p(a[i]), a.shape[1], _p(codes[i]))
    return codes, scales


# ---------------------------------------------------------------- RAGGED extend

def topk_ragged(logits, row_len, row_to_req, req_offset, topk: int, rows: Optional[Sequence[int]] = None):
    """indices int32 [len(rows), topk]: top-k positions of each row plus its
    request's offset in the flattened KV (ascending, -1 padded)."""
    lib = _load()
    lg = _c(logits, np.float32)
    rl = _c(row_len, np.int32)
    r2q = _c(row_to_req, np.int32)
    off = _c(req_offset, np.int32)
    rows = list(range(len(rl))) if rows is None else list(rows)
    out = np.zeros((len(rows), topk), dtype=np.int32)
    for i, r in enumerate(rows):
        L = int(rl[r])
        lp = C.c_void_p(lg.ctypes.data + r * lg.shape[1] * 4)
        op = C.c_void_p(out.ctypes.data + i * topk * 4)
        lib.orc_topk_ragged_row(lp, L, topk, int(off[int(r2q[r])]), op)
    return out


def flatten_page_table(page_table_1, kv_len) -> np.ndarray:
    lib = _load()
    pt = _c(page_table_1, np.int32)
    kl = _c(kv_len, np.int32)
    out = np.zeros((max(1, int(kl.sum())),), dtype=np.int32)
    n = lib.orc_flatten_page_table(len(kl), _p(pt), pt.shape[1], _p(kl), _p(out))
    return out[:n]


# ---------------------------------------------------------------- chunk-local attention

def local_attention(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, sm_scale: float):
    """q bf16 bits [total_q, Hq, D]; caches bf16 bits [pages, ps, Hkv, D]; block_table int32
    [nvb, bt_ld]; cu_seqlens_q [nvb + 1]; seqused_k [nvb].  Returns (out [total_q, Hq, D],
    lse [total_q, Hq]) in float64."""
    lib = _load()
    qq = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_table, np.int32)
    cq = _c(cu_seqlens_q, np.int32)
    sk = _c(seqused_k, np.int32)
    total, Hq, D = qq.shape
    num_pages, ps, Hkv, _ = kc.shape
    out = np.zeros((total, Hq, D), dtype=np.float64)
    lse = np.zeros((total, Hq), dtype=np.float64)
    for b in range(len(sk)):
        for i in range(int(cq[b + 1] - cq[b])):
            t = int(cq[b]) + i
            rc = lib.orc_local_attention_row(b, i, Hq, Hkv, D, ps, num_pages, _p(bt), bt.shape[1], _p(cq), _p(sk),
                                             _p(qq[t]), _p(kc), _p(vc), float(sm_scale),
                                             C.c_void_p(out.ctypes.data + t * Hq * D * 8),
                                             C.c_void_p(lse.ctypes.data + t * Hq * 8))
            if rc != 0:
                raise ValueError("page id out of range")
    return out, lse
