"""Seeded synthetic inputs for the sparse-attention decode/extend path.

This module only draws random numbers and lays them out in the storage
formats the path consumes (e4m3 / bfloat16 / float32 buffers, a paged
request-to-token table).  It holds none of the path's arithmetic: no
metadata, no scores, no selection, no attention.  Both the CUDA path and the
oracle are fed from here, and nothing here depends on either of them.

Encodings use PyTorch's own dtype casts (round-to-nearest-even), so the bytes
are reproducible on any host with the same NumPy / PyTorch versions.
Random draws are chunked with one NumPy generator per chunk (spawned from the
config seed), so results do not depend on the number of worker threads.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

MODE_DECODE, MODE_EXTEND, MODE_VERIFY = 0, 1, 2
DT_F32, DT_BF16, DT_E4M3 = 0, 1, 2
E4M3_MAX = 448.0
_CHUNK = 1 << 22  # elements per independent random stream
_SLOT_BLOCK = 1 << 16  # KV / K rows drawn and encoded per block


@dataclass
class Workload:
    name: str
    mode: int
    B: int
    seq_lens: np.ndarray  # int32 [B]; committed tokens (extend: including new ones)
    extend_lens: Optional[np.ndarray]  # int32 [B] (extend only)
    n_draft: int
    topk: int
    page_size: int
    Hi: int
    Di: int
    idx_dtype: int  # DT_E4M3 or DT_F32
    H: int
    d_latent: int
    d_rope: int
    q_dtype: int  # DT_BF16 or DT_F32
    kv_dtype: int  # DT_BF16, DT_E4M3 or DT_F32
    sm_scale: float
    R: int  # query rows of the step
    W: int  # page-table width: the longest cache length of the step
    num_pages: int
    req_to_token: np.ndarray  # int32 [pool_rows, W_pool]
    req_pool_indices: np.ndarray  # int32 [B]
    q_idx: np.ndarray  # uint8 e4m3 [R,Hi,Di] or float32
    weights: np.ndarray  # float32 [R,Hi]
    k_cache: np.ndarray  # uint8 e4m3 [num_pages, ps, Di] or float32
    k_scale: np.ndarray  # float32 [num_pages, ps]
    q_nope: np.ndarray  # uint16 (bf16 bits) [R,H,d_latent] or float32
    q_rope: np.ndarray  # uint16 [R,H,d_rope] or float32
    kv: np.ndarray  # bf16 bits [slots, d_latent+d_rope] | uint8 [slots, row_bytes] | float32
    extra: dict = field(default_factory=dict)

    @property
    def cache_lens(self) -> np.ndarray:
        """Per-request number of cached tokens the step's page table covers."""
        return self.seq_lens + (self.n_draft if self.mode == MODE_VERIFY else 0)

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.page_size

    @property
    def kv_row_bytes(self) -> int:
        if self.kv_dtype == DT_E4M3:
            return self.d_latent + 4 * (self.d_latent // 128) + 2 * self.d_rope
        return (self.d_latent + self.d_rope) * (4 if self.kv_dtype == DT_F32 else 2)


# --------------------------------------------------------------------------
# random draws
# --------------------------------------------------------------------------

def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _draw(seed_seq: np.random.SeedSequence, n: int, kind: str, **kw) -> np.ndarray:
    """n float32 draws, generated in fixed chunks with one stream per chunk."""
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    seqs = seed_seq.spawn(nchunks)
    out = np.empty(n, dtype=np.float32)

    def fill(i):
        g = np.random.default_rng(seqs[i])
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        if kind == "normal":
            g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        else:
            out[lo:hi] = g.uniform(kw.get("low", 0.0), kw.get("high", 1.0), hi - lo).astype(np.float32)

    if nchunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def _to_e4m3(x: np.ndarray) -> np.ndarray:
    """float32 -> e4m3 bytes (torch cast, round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _to_bf16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _e4m3_rows_with_scale(x: np.ndarray, block: int):
    """Scale each `block`-long run of the last axis by amax/448 and encode it.

    Returns (codes uint8 same shape, scales float32 [..., n_blocks]).  A block
    of zeros gets scale 1.
    """
    shp = x.shape
    xb = x.reshape(-1, shp[-1] // block, block)
    amax = np.abs(xb).max(axis=-1)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)
    codes = _to_e4m3((xb / scale[..., None]).astype(np.float32))
    return codes.reshape(shp), scale.reshape(shp[:-1] + (shp[-1] // block,))


# --------------------------------------------------------------------------
# page tables
# --------------------------------------------------------------------------

def _paged_tables(rng: np.random.Generator, cache_lens: np.ndarray, ps: int, slack: float):
    """Random page placement: every request owns whole pages, the pages of all
    requests are a random permutation of the physical page pool.

    Returns (req_to_token [pool_rows, W_pool], req_pool_indices [B], num_pages, W).
    Entries past a request's length are 0, as in a zero-initialised pool.
    """
    B = len(cache_lens)
    pages_per = [(int(l) + ps - 1) // ps for l in cache_lens]
    used = sum(pages_per)
    num_pages = used + max(1, int(math.ceil(used * slack)))
    perm = rng.permutation(num_pages).astype(np.int64)
    W = int(cache_lens.max()) if B else 0
    W_pool = ((W + ps - 1) // ps) * ps + ps
    pool_rows = B + 2
    r2t = np.zeros((pool_rows, W_pool), dtype=np.int32)
    rows = rng.permutation(pool_rows)[:B].astype(np.int32)
    off = 0
    for b in range(B):
        pg = perm[off: off + pages_per[b]]
        off += pages_per[b]
        t = np.arange(int(cache_lens[b]), dtype=np.int64)
        r2t[rows[b], : len(t)] = (pg[t // ps] * ps + t % ps).astype(np.int32)
    return r2t, rows, num_pages, W


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

def make_workload(name: str, *, mode: int, seq_lens, extend_lens=None, n_draft: int = 0,
                  topk: int, page_size: int, Hi: int, Di: int, idx_dtype: int, H: int,
                  d_latent: int, d_rope: int, q_dtype: int, kv_dtype: int, sm_scale: float,
                  seed: int, weight_dist: str = "normal8", kv_outliers: float = 0.0,
                  slack: float = 0.01) -> Workload:
    """Draw one step's inputs.

    Distributions: q_idx, K, q, KV ~ N(0,1); weights N(0,1)/8 ("normal8") or
    U(0,1) ("uniform"); optional KV outliers: that fraction of latent elements
    multiplied by 20.  e4m3 K rows carry one float32 scale (amax/448); e4m3 KV
    rows carry one float32 scale per 128 latent elements (amax/448); the rope
    part stays bfloat16.  float32 configs use k_scale = 1.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = len(seq_lens)
    ext = None if extend_lens is None else np.asarray(extend_lens, dtype=np.int32)
    if mode == MODE_DECODE:
        R = B
    elif mode == MODE_VERIFY:
        R = B * n_draft
    else:
        R = int(ext.sum())
    cache = seq_lens + (n_draft if mode == MODE_VERIFY else 0)

    root = np.random.SeedSequence(seed)
    s_tab, s_q, s_w, s_k, s_qm, s_kv, s_out = root.spawn(7)
    rng_tab = np.random.default_rng(s_tab)
    r2t, rows, num_pages, W = _paged_tables(rng_tab, cache, page_size, slack)
    slots = num_pages * page_size

    # indexer inputs
    qi = _draw(s_q, R * Hi * Di, "normal").reshape(R, Hi, Di)
    if weight_dist == "uniform":
        w = _draw(s_w, R * Hi, "uniform", low=0.0, high=1.0).reshape(R, Hi)
    else:
        w = (_draw(s_w, R * Hi, "normal") / np.float32(8.0)).reshape(R, Hi)
    if idx_dtype == DT_E4M3:
        q_idx = _to_e4m3(qi)
        k_cache = np.empty((slots, Di), dtype=np.uint8)
        k_scale = np.empty((slots,), dtype=np.float32)
    else:
        q_idx = qi
        k_cache = np.empty((slots, Di), dtype=np.float32)
        k_scale = np.ones((slots,), dtype=np.float32)
    del qi
    k_blocks = (slots + _SLOT_BLOCK - 1) // _SLOT_BLOCK
    for i, sq in enumerate(s_k.spawn(max(1, k_blocks))):
        lo, hi = i * _SLOT_BLOCK, min(slots, (i + 1) * _SLOT_BLOCK)
        if lo >= hi:
            break
        k = _draw(sq, (hi - lo) * Di, "normal").reshape(hi - lo, Di)
        if idx_dtype == DT_E4M3:
            codes, sc = _e4m3_rows_with_scale(k, Di)
            k_cache[lo:hi], k_scale[lo:hi] = codes, sc[:, 0]
        else:
            k_cache[lo:hi] = k
    k_cache = k_cache.reshape(num_pages, page_size, Di)
    k_scale = k_scale.reshape(num_pages, page_size)

    # attention inputs
    dq = d_latent + d_rope
    qm = _draw(s_qm, R * H * dq, "normal").reshape(R, H, dq)
    if q_dtype == DT_BF16:
        q_nope, q_rope = _to_bf16(qm[..., :d_latent]), _to_bf16(qm[..., d_latent:])
    else:
        q_nope, q_rope = np.ascontiguousarray(qm[..., :d_latent]), np.ascontiguousarray(qm[..., d_latent:])
    del qm
    nb = d_latent // 128
    if kv_dtype == DT_E4M3:
        kv = np.empty((slots, d_latent + 4 * nb + 2 * d_rope), dtype=np.uint8)
    else:
        kv = np.empty((slots, dq), dtype=np.uint16 if kv_dtype == DT_BF16 else np.float32)
    kv_blocks = (slots + _SLOT_BLOCK - 1) // _SLOT_BLOCK
    for i, (sq, so) in enumerate(zip(s_kv.spawn(max(1, kv_blocks)), s_out.spawn(max(1, kv_blocks)))):
        lo, hi = i * _SLOT_BLOCK, min(slots, (i + 1) * _SLOT_BLOCK)
        if lo >= hi:
            break
        n = hi - lo
        kvf = _draw(sq, n * dq, "normal").reshape(n, dq)
        if kv_outliers > 0.0:
            g = np.random.default_rng(so)
            n_out = int(round(kv_outliers * n * d_latent))
            flat = g.choice(n * d_latent, size=n_out, replace=False)
            lat = np.ascontiguousarray(kvf[:, :d_latent]).reshape(-1)
            lat[flat] *= np.float32(20.0)
            kvf[:, :d_latent] = lat.reshape(n, d_latent)
        if kv_dtype == DT_BF16:
            kv[lo:hi] = _to_bf16(kvf)
        elif kv_dtype == DT_F32:
            kv[lo:hi] = kvf
        else:
            codes, sc = _e4m3_rows_with_scale(kvf[:, :d_latent], 128)
            kv[lo:hi, :d_latent] = codes
            kv[lo:hi, d_latent: d_latent + 4 * nb] = np.ascontiguousarray(sc, dtype=np.float32).view(np.uint8).reshape(n, 4 * nb)
            kv[lo:hi, d_latent + 4 * nb:] = _to_bf16(kvf[:, d_latent:]).view(np.uint8).reshape(n, 2 * d_rope)
        del kvf

    return Workload(name=name, mode=mode, B=B, seq_lens=seq_lens, extend_lens=ext,
                    n_draft=n_draft, topk=topk, page_size=page_size, Hi=Hi, Di=Di,
                    idx_dtype=idx_dtype, H=H, d_latent=d_latent, d_rope=d_rope,
                    q_dtype=q_dtype, kv_dtype=kv_dtype, sm_scale=float(sm_scale), R=R, W=W,
                    num_pages=num_pages, req_to_token=r2t, req_pool_indices=rows,
                    q_idx=q_idx, weights=w.astype(np.float32), k_cache=k_cache,
                    k_scale=k_scale.astype(np.float32), q_nope=q_nope, q_rope=q_rope, kv=kv)


SM_SCALE_V32 = 192 ** -0.5


def config(name: str, seed: Optional[int] = None, *, scale: float = 1.0) -> Workload:
    """The five named workloads of the method (full size by default).

    `scale` < 1 shrinks batch and lengths proportionally for quick tests while
    keeping every other property (paging, dtypes, head counts, topk).
    """
    def rng_for(s):
        return np.random.default_rng(np.random.SeedSequence([s, 1234]))

    if name == "tiny_fp32_decode":
        return make_workload(name, mode=MODE_DECODE, seq_lens=[64, 100], topk=32, page_size=16,
                             Hi=4, Di=32, idx_dtype=DT_F32, H=4, d_latent=64, d_rope=16,
                             q_dtype=DT_F32, kv_dtype=DT_F32, sm_scale=80 ** -0.5,
                             seed=0 if seed is None else seed, weight_dist="uniform")
    if name == "v32_decode_bf16":
        seed = 2 if seed is None else seed
        B = max(1, int(round(32 * scale)))
        lo, hi = max(64, int(4096 * scale)), max(128, int(32768 * scale))
        L = rng_for(seed).integers(lo, hi + 1, size=B)
        return make_workload(name, mode=MODE_DECODE, seq_lens=L, topk=2048, page_size=64,
                             Hi=64, Di=128, idx_dtype=DT_E4M3, H=128, d_latent=512, d_rope=64,
                             q_dtype=DT_BF16, kv_dtype=DT_BF16, sm_scale=SM_SCALE_V32, seed=seed)
    if name == "fp8kv_decode_h16":
        seed = 3 if seed is None else seed
        B = max(1, int(round(128 * scale)))
        L = np.full(B, max(64, int(8192 * scale)), dtype=np.int32)
        return make_workload(name, mode=MODE_DECODE, seq_lens=L, topk=2048, page_size=64,
                             Hi=64, Di=128, idx_dtype=DT_E4M3, H=16, d_latent=512, d_rope=64,
                             q_dtype=DT_BF16, kv_dtype=DT_E4M3, sm_scale=SM_SCALE_V32, seed=seed,
                             kv_outliers=0.01)
    if name == "chunked_extend":
        seed = 4 if seed is None else seed
        nb = 4
        new = max(16, int(2048 * scale))
        prefix = max(16, int(8192 * scale))
        return make_workload(name, mode=MODE_EXTEND, seq_lens=[prefix + new] * nb,
                             extend_lens=[new] * nb, topk=2048, page_size=64, Hi=64, Di=128,
                             idx_dtype=DT_E4M3, H=128, d_latent=512, d_rope=64, q_dtype=DT_BF16,
                             kv_dtype=DT_BF16, sm_scale=SM_SCALE_V32, seed=seed)
    if name == "verify_long_fp8kv":
        seed = 5 if seed is None else seed
        B = max(1, int(round(64 * scale)))
        lo, hi = max(64.0, 16384 * scale), max(128.0, 131072 * scale)
        u = rng_for(seed).uniform(math.log(lo), math.log(hi), size=B)
        L = np.floor(np.exp(u)).astype(np.int32)
        return make_workload(name, mode=MODE_VERIFY, seq_lens=L, n_draft=4, topk=2048,
                             page_size=64, Hi=64, Di=128, idx_dtype=DT_E4M3, H=128, d_latent=512,
                             d_rope=64, q_dtype=DT_BF16, kv_dtype=DT_E4M3, sm_scale=SM_SCALE_V32,
                             seed=seed)
    raise KeyError(name)


CONFIG_NAMES = ["tiny_fp32_decode", "v32_decode_bf16", "fp8kv_decode_h16", "chunked_extend",
                "verify_long_fp8kv"]


# --------------------------------------------------------------------------
# chunk-local dense attention (the second workload)
# --------------------------------------------------------------------------

@dataclass
class LocalAttnWorkload:
    name: str
    chunk: int                 # attention chunk size (a multiple of page_size)
    page_size: int
    Hq: int
    Hkv: int
    D: int
    seq_lens: np.ndarray       # int32 [B]: keys of each request, new queries included
    q_lens: np.ndarray         # int32 [B]: new query rows (the last q_lens[b] positions)
    cu_seqlens_q: np.ndarray   # int32 [B + 1]: query row start of each request
    block_table: np.ndarray    # int32 [B, W]: page ids; W covers each request's last chunk
    q: np.ndarray              # bf16 bits [total_q, Hq, D]
    k_cache: np.ndarray        # bf16 bits [num_pages, page_size, Hkv, D]
    v_cache: np.ndarray        # bf16 bits [num_pages, page_size, Hkv, D]
    sm_scale: float

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])


def make_local_attention(name: str, *, seq_lens, q_lens, chunk: int, Hq: int, Hkv: int, D: int,
                         page_size: int, seed: int, slack: float = 0.02) -> LocalAttnWorkload:
    """Requests own whole pages of a randomly permuted page pool; q, K and V are
    standard normal values rounded to bfloat16.  Block-table columns past a
    request's pages hold page 0 (never read: they lie past the request's keys)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    assert chunk % page_size == 0 and np.all(q_lens >= 1) and np.all(q_lens <= seq_lens)
    rng = np.random.default_rng(np.random.SeedSequence([seed, 77]))
    ps = page_size
    pages_per = (seq_lens.astype(np.int64) + ps - 1) // ps
    used = int(pages_per.sum())
    num_pages = used + max(1, int(math.ceil(used * slack)))
    perm = rng.permutation(num_pages).astype(np.int32)
    W = int(max((int(L) + chunk - 1) // chunk * (chunk // ps) for L in seq_lens))
    bt = np.zeros((len(seq_lens), W), dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[off: off + n]
        off += int(n)
    cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    total_q = int(cu[-1])
    q_ss, k_ss, v_ss = np.random.SeedSequence([seed, 78]).spawn(3)
    shape = (num_pages, ps, Hkv, D)
    n = num_pages * ps * Hkv * D
    q = _to_bf16(_draw(q_ss, total_q * Hq * D, "normal")).reshape(total_q, Hq, D)
    k = _to_bf16(_draw(k_ss, n, "normal")).reshape(shape)
    v = _to_bf16(_draw(v_ss, n, "normal")).reshape(shape)
    return LocalAttnWorkload(name, chunk, ps, Hq, Hkv, D, seq_lens, q_lens, cu, bt, q, k, v, D ** -0.5)


def local_config(name: str, seed: Optional[int] = None, *, scale: float = 1.0) -> LocalAttnWorkload:
    """Named chunk-local attention workloads.

    local_decode_c8192: 32 decoding requests (one new query each) whose lengths
    are uniform in [1, 16384], attention chunk 8192, 40 query heads over 8
    key/value heads of 128 dims, pages of 64 tokens: each query attends to the
    1..8192 keys of its current chunk.  `scale` < 1 shrinks the batch and the
    lengths (chunk included) for quick tests."""
    if name == "local_decode_c8192":
        seed = 6 if seed is None else seed
        rng = np.random.default_rng(np.random.SeedSequence([seed, 1234]))
        B = max(1, int(round(32 * scale)))
        chunk = max(64, int(8192 * scale) // 64 * 64)
        L = rng.integers(1, 2 * chunk + 1, size=B)
        return make_local_attention(name, seq_lens=L, q_lens=np.ones(B, np.int32), chunk=chunk, Hq=40,
                                    Hkv=8, D=128, page_size=64, seed=seed)
    raise KeyError(name)


LOCAL_CONFIG_NAMES = ["local_decode_c8192"]
