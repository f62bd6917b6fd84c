"""Shared helpers of the parity tests: run the CUDA path through the C ABI and
compare each stage with the oracle on the same seeded inputs."""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

import oracle
import workloads as W

# Tolerances (the method's stated bars):
#   metadata, indices: bit-exact
#   logits: |g - o| <= 1e-3 * (|o| + rms of the oracle row)   (fp8 in, fp32 accumulate)
#   out, lse: |g - o| <= tol * (1 + |o|), tol = 2e-2 bf16 KV, 6e-2 fp8 KV, 1e-4 fp32
LOGIT_RTOL = 1e-3


def attn_tol(wl) -> float:
    if wl.kv_dtype == W.DT_F32:
        return 1e-4
    return 6e-2 if wl.kv_dtype == W.DT_E4M3 else 2e-2


def oracle_metadata(wl):
    return oracle.metadata(wl.mode, wl.seq_lens, wl.req_to_token, wl.req_pool_indices, W=wl.W,
                           topk=wl.topk, page_size=wl.page_size, extend_lens=wl.extend_lens,
                           n_draft=wl.n_draft)


def check_metadata(step, md_o):
    for k in ["cache_seqlens", "cu_seqlens_k", "cu_seqlens_q", "seqlens_expanded", "nsa_cache_seqlens",
              "nsa_cu_seqlens_k", "nsa_cu_seqlens_q", "row_to_req", "indexer_ks", "indexer_ke"]:
        if k not in md_o:
            continue
        g = step.md[k].cpu().numpy()
        assert np.array_equal(g, md_o[k]), f"metadata {k} differs"
    if "page_table_1" in step.md:
        g = step.md["page_table_1"].cpu().numpy()[:, : step.W]
        assert np.array_equal(g, md_o["page_table_1"]), "page_table_1 differs"
    if "req_rows" in step.md:
        assert np.array_equal(step.md["req_rows"].cpu().numpy(), step.req_pool_indices.cpu().numpy()), \
            "req_rows differs from req_pool_indices"
    npg = md_o["real_page_table"].shape[1]
    g = step.md["real_page_table"].cpu().numpy()[:, :npg]
    assert np.array_equal(g, md_o["real_page_table"]), "real_page_table differs"


def check_logits(g_rows: np.ndarray, o_rows: np.ndarray, lens: np.ndarray):
    for i, L in enumerate(lens):
        g, o = g_rows[i, :L].astype(np.float64), o_rows[i, :L].astype(np.float64)
        rms = np.sqrt(np.mean(o ** 2)) if L else 0.0
        err = np.abs(g - o) - LOGIT_RTOL * (np.abs(o) + rms)
        assert np.all(err <= 0), f"logits row {i}: worst excess {err.max():.3e} (L={L})"


def check_attention(out_g: np.ndarray, lse_g: np.ndarray, out_o: np.ndarray, lse_o: np.ndarray, tol: float):
    og = out_g.astype(np.float64)
    bad = np.abs(og - out_o) > tol * (1.0 + np.abs(out_o))
    assert not bad.any(), f"out: {bad.sum()} elements beyond tol {tol}, max err {np.abs(og - out_o).max():.3e}"
    fin = np.isfinite(lse_o)
    assert np.array_equal(np.isfinite(lse_g), fin), "lse finiteness differs"
    assert np.array_equal(lse_g[~fin], lse_o[~fin])
    bad = np.abs(lse_g[fin] - lse_o[fin]) > tol * (1.0 + np.abs(lse_o[fin]))
    assert not bad.any(), f"lse: {bad.sum()} beyond tol, max err {np.abs(lse_g[fin] - lse_o[fin]).max():.3e}"


def host_digit_hist(lg_rows: np.ndarray, lens) -> np.ndarray:
    """Per row, counts of the leading 11 bits of each score's order-preserving
    32-bit key (NaN lowest, -0 == +0, negative scores bit-reversed below the
    positive ones): the digit histogram nsa_indexer_logits accumulates."""
    out = np.zeros((len(lens), 2048), np.int64)
    for i, L in enumerate(lens):
        x = np.ascontiguousarray(lg_rows[i, :L], dtype=np.float32)
        u = x.view(np.uint32).astype(np.uint64)
        key = np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)
        key = np.where(((u << 1) & 0xFFFFFFFF) == 0, 0x80000000, key)
        key = np.where(np.isnan(x), 0, key)
        out[i] = np.bincount((key >> 21).astype(np.int64), minlength=2048)
    return out


def check_digit_hist(step, rows, lg_rows: np.ndarray, lens):
    """The indexer's digit counts equal those of the logits it wrote."""
    if getattr(step, "score_hist", None) is None:
        return
    hg = step.score_hist.cpu().numpy().view(np.uint32)[rows].astype(np.int64)
    exp = host_digit_hist(lg_rows, lens)
    bad = np.nonzero((hg != exp).any(axis=1))[0]
    assert len(bad) == 0, f"indexer digit counts differ from its logits in rows {[rows[i] for i in bad[:5]]}"


def out_to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def sample_rows(wl, n: int, seed: int = 0) -> list:
    """First, last and n-2 random rows (sorted, distinct)."""
    if wl.R <= n:
        return list(range(wl.R))
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, wl.R - 1), size=max(0, n - 2), replace=False)
    return sorted(set([0, wl.R - 1] + [int(x) for x in mid]))


def full_parity(step, wl, rows: Optional[Sequence[int]] = None, e2e: bool = True,
                e2e_topk_rows: Optional[Sequence[int]] = None):
    """Stage-by-stage parity on `rows` (all rows by default) plus the end-to-end
    check; the end-to-end top-k check (GPU indices == exact top-k of the GPU
    logits) runs on `e2e_topk_rows` (default: `rows`).  Asserts on any mismatch."""
    rows = list(range(wl.R)) if rows is None else list(rows)
    e2e_topk_rows = rows if e2e_topk_rows is None else list(e2e_topk_rows)
    md_o = oracle_metadata(wl)
    step.metadata()
    torch.cuda.synchronize()
    check_metadata(step, md_o)

    # indexer
    step.indexer()
    torch.cuda.synchronize()
    lens = md_o["seqlens_expanded"][rows]
    lo = oracle.indexer_logits(wl.idx_dtype, wl.q_idx, wl.weights, wl.k_cache, wl.k_scale,
                               md_o["real_page_table"], md_o["row_to_req"], md_o["seqlens_expanded"],
                               rows=rows, width=wl.W)
    lg = step.logits.cpu().numpy()[rows]
    check_logits(lg, lo, lens)
    check_digit_hist(step, rows, lg, lens)

    # top-k fed the oracle's logits (bit-exact)
    feed = torch.full_like(step.logits, float("nan"))
    lo_full = np.nan_to_num(lo, nan=0.0)
    feed[torch.as_tensor(rows, device=feed.device), : wl.W] = torch.from_numpy(lo_full).to(feed.device)
    step.topk_transform(logits=feed)
    torch.cuda.synchronize()
    io = oracle.topk_transform(lo_full, md_o["seqlens_expanded"], md_o["row_to_req"], md_o["page_table_1"],
                               wl.topk, rows=rows, logits_rows_are_subset=True)
    ig = step.indices.cpu().numpy()[rows]
    assert np.array_equal(ig, io), "top-k indices (fed the oracle's logits) differ"

    # attention fed the oracle's indices
    idx_feed = torch.full_like(step.indices, -1)
    idx_feed[torch.as_tensor(rows, device=idx_feed.device)] = torch.from_numpy(io).to(idx_feed.device)
    step.attention(indices=idx_feed)
    torch.cuda.synchronize()
    oo, lso = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, io, wl.sm_scale,
                                rows=rows, indices_rows_are_subset=True)
    check_attention(out_to_np(step.out)[rows], step.lse.cpu().numpy()[rows], oo, lso, attn_tol(wl))
    assert step.status_code() == 0

    if e2e:
        # whole step on the GPU; the GPU's indices must be the exact top-k of
        # the GPU's logits, and attention over them must match the oracle.
        step.run()
        torch.cuda.synchronize()
        lg_all = step.logits.cpu().numpy()
        lg = lg_all[rows]
        check_logits(lg, lo, lens)
        ig_all = step.indices.cpu().numpy()
        lg_t = lg_all[e2e_topk_rows]
        io2 = oracle.topk_transform(lg_t, md_o["seqlens_expanded"], md_o["row_to_req"], md_o["page_table_1"],
                                    wl.topk, rows=e2e_topk_rows, logits_rows_are_subset=True)
        bad = np.nonzero((ig_all[e2e_topk_rows] != io2).any(axis=1))[0]
        assert len(bad) == 0, (f"end-to-end indices are not the top-k of the GPU logits in rows "
                               f"{[e2e_topk_rows[i] for i in bad[:5]]}")
        if getattr(step, "score_hist", None) is not None:
            assert not step.score_hist.any().item(), "the top-k left digit counts behind"
        ig = ig_all[rows]
        oo2, lso2 = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, ig, wl.sm_scale,
                                      rows=rows, indices_rows_are_subset=True)
        check_attention(out_to_np(step.out)[rows], step.lse.cpu().numpy()[rows], oo2, lso2, attn_tol(wl))
        assert step.status_code() == 0
