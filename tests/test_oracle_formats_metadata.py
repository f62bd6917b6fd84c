"""Pins of the oracle's number formats and per-step metadata (CPU only).

Each check ties the oracle to something other than itself: values fixed by the
format definitions, PyTorch's own dtype conversions, worked examples printed
on the pages (tests/golden), closed forms and brute force.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.golden import load
import workloads as W


# ------------------------------------------------------------------ formats

def test_e4m3_values_fixed_by_the_format():
    # OCP E4M3FN: bias 7, 3 mantissa bits, subnormals below 2^-6, no infinities,
    # S.1111.111 = NaN, largest finite 448.
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xB8: -1.0, 0xFE: -448.0}
    got = oracle.e4m3_to_f64(np.array(list(table), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(table.values())))
    nan = oracle.e4m3_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(nan).all()
    neg0 = oracle.e4m3_to_f64(np.array([0x80], dtype=np.uint8))[0]
    assert neg0 == 0.0 and math.copysign(1.0, neg0) < 0


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_bf16_matches_torch():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite values
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_to_f64(bits), ref)


# ------------------------------------------------------------------ metadata

def _pool(rng, cache_lens, ps, extra_cols=0):
    r2t, rows, num_pages, Wd = W._paged_tables(rng, np.asarray(cache_lens, np.int32), ps, 0.05)
    return r2t, rows, Wd


def test_indexer_k_start_end_worked_example():
    g = load("indexer_k_start_end_worked_example.txt")
    rng = np.random.default_rng(0)
    r2t, rpi, Wd = _pool(rng, g["seq_lens"], 1)
    md = oracle.metadata(W.MODE_EXTEND, g["seq_lens"], r2t, rpi, W=Wd, topk=2048, page_size=1,
                         extend_lens=g["extend_lens"])
    assert np.array_equal(md["indexer_ks"], g["ks"])
    assert np.array_equal(md["indexer_ke"], g["ke"])


@pytest.mark.parametrize("mode", [W.MODE_DECODE, W.MODE_VERIFY, W.MODE_EXTEND])
@pytest.mark.parametrize("ps", [1, 16, 64])
def test_metadata_closed_forms(mode, ps):
    rng = np.random.default_rng(100 + mode * 10 + ps)
    B, n, topk = 7, 3, 40
    seq = rng.integers(1, 300, size=B).astype(np.int32)
    ext = np.minimum(seq, rng.integers(1, 60, size=B)).astype(np.int32) if mode == W.MODE_EXTEND else None
    cache = seq + (n if mode == W.MODE_VERIFY else 0)
    r2t, rpi, Wd = _pool(rng, cache, ps)
    md = oracle.metadata(mode, seq, r2t, rpi, W=Wd, topk=topk, page_size=ps, extend_lens=ext,
                         n_draft=n if mode == W.MODE_VERIFY else 0)
    R = md["R"]
    assert np.array_equal(md["cache_seqlens"], cache)
    assert np.array_equal(md["cu_seqlens_k"], np.concatenate([[0], np.cumsum(cache)]))
    if mode == W.MODE_DECODE:
        assert R == B
        assert np.array_equal(md["seqlens_expanded"], cache)
        assert np.array_equal(md["cu_seqlens_q"], np.arange(B + 1))
        assert np.array_equal(md["row_to_req"], np.arange(B))
    elif mode == W.MODE_VERIFY:
        # target-verify: n draft rows per request see seq+1 ... seq+n tokens
        assert R == B * n
        assert np.array_equal(md["seqlens_expanded"].reshape(B, n), seq[:, None] + np.arange(1, n + 1))
        assert np.array_equal(md["cu_seqlens_q"], np.arange(R + 1))
        assert np.array_equal(md["row_to_req"], np.repeat(np.arange(B), n))
    else:
        assert R == ext.sum()
        assert np.array_equal(md["cu_seqlens_q"], np.concatenate([[0], np.cumsum(ext)]))
        exp = np.concatenate([np.arange(c - e + 1, c + 1) for c, e in zip(cache, ext)])
        assert np.array_equal(md["seqlens_expanded"], exp)
        assert np.array_equal(md["row_to_req"], np.repeat(np.arange(B), ext))
        ks = np.repeat(np.concatenate([[0], np.cumsum(seq)[:-1]]), ext)
        assert np.array_equal(md["indexer_ks"], ks)
        assert np.array_equal(md["indexer_ke"], ks + exp)
    # lengths clipped to topk and their cumulative sum (the per-row sparse
    # lengths and their offsets)
    clipped = np.minimum(md["seqlens_expanded"], topk)
    assert np.array_equal(md["nsa_cache_seqlens"], clipped)
    assert np.array_equal(md["nsa_cu_seqlens_k"], np.concatenate([[0], np.cumsum(clipped)]))
    assert np.array_equal(md["nsa_cu_seqlens_q"], np.arange(R + 1))
    # page tables: a gather of req_to_token, and its page-granular view
    assert np.array_equal(md["page_table_1"], r2t[rpi, :Wd])
    pt = md["page_table_1"]
    rpt = md["real_page_table"]
    if ps == 1:
        assert np.array_equal(rpt, pt)
    for b in range(B):
        t = np.arange(cache[b])
        assert np.array_equal(pt[b, t], rpt[b, t // ps] * ps + t % ps)


def test_metadata_named_workload_rows():
    # chunked extend: 4 x (8192 prefix + 2048 new) -> rows see 8193 ... 10240
    wl = W.config("chunked_extend")
    md = oracle.metadata(wl.mode, wl.seq_lens, wl.req_to_token, wl.req_pool_indices, W=wl.W,
                         topk=wl.topk, page_size=wl.page_size, extend_lens=wl.extend_lens)
    assert md["R"] == 8192
    assert np.array_equal(md["seqlens_expanded"], np.tile(np.arange(8193, 10241), 4))
    assert np.all(md["nsa_cache_seqlens"] == 2048)


def test_metadata_rejects_length_beyond_table():
    rng = np.random.default_rng(3)
    r2t, rpi, Wd = _pool(rng, [10, 20], 4)
    with pytest.raises(ValueError):
        oracle.metadata(W.MODE_DECODE, np.array([10, 20]), r2t, rpi, W=Wd - 1, topk=8, page_size=4)


# ------------------------------------------------------------------ local attention

def test_local_virtual_batches_worked_example():
    g = load("local_virtual_batches_worked_example.txt")
    bt = g["block_table"].reshape(int(g["block_table_rows"][0]), int(g["block_table_cols"][0]))
    sq, cu, sk, st, btl = oracle.local_virtual_batches(int(g["attn_chunk_size"][0]),
                                                       int(g["page_size"][0]), g["query_start_loc"],
                                                       g["seq_lens"], bt)
    assert np.array_equal(sq, g["seqlens_q_local"])
    assert np.array_equal(cu, g["cu_seqlens_q_local"])
    assert np.array_equal(sk, g["seqlens_k_local"])
    assert np.array_equal(st, g["k_seqstarts_absolute"])
    assert np.array_equal(btl.reshape(-1), g["block_table_local"])
    # the page's intermediate values: virtual batches per request and the
    # queries of each request's first virtual batch
    blocks = g["local_blocks"]
    first = np.concatenate([[0], np.cumsum(blocks)[:-1]])
    assert len(sq) == blocks.sum()
    assert np.array_equal(np.add.reduceat(sq, first), np.diff(g["query_start_loc"]))
    assert np.array_equal(sq[first], g["q_tokens_in_first_block"])


def _brute_force_local(c, ps, q_lens, kv_lens, bt):
    """Group every query token by the attention chunk of its own position."""
    sq, sk, st, btl = [], [], [], []
    for b, (q, kv) in enumerate(zip(q_lens, kv_lens)):
        pos = np.arange(kv - q, kv)
        for ch in np.unique(pos // c):
            sq.append(int(np.sum(pos // c == ch)))
            start = int(ch * c)
            st.append(start)
            sk.append(min(kv, start + c) - start)
            btl.append(bt[b, start // ps: start // ps + c // ps])
    return (np.array(sq), np.array(sk), np.array(st), np.array(btl))


@pytest.mark.parametrize("seed", range(6))
def test_local_virtual_batches_brute_force(seed):
    rng = np.random.default_rng(seed)
    ps = int(rng.choice([1, 2, 4]))
    c = ps * int(rng.integers(1, 5))
    B = int(rng.integers(1, 6))
    kv = rng.integers(1, 40, size=B)
    q = np.array([int(rng.integers(1, k + 1)) for k in kv])
    cq = np.concatenate([[0], np.cumsum(q)])
    cols = (int(kv.max()) + c) // ps + 2
    bt = rng.integers(0, 1000, size=(B, cols)).astype(np.int32)
    sq, cu, sk, st, btl = oracle.local_virtual_batches(c, ps, cq, kv, bt)
    e_sq, e_sk, e_st, e_btl = _brute_force_local(c, ps, q, kv, bt)
    assert np.array_equal(sq, e_sq) and np.array_equal(sk, e_sk) and np.array_equal(st, e_st)
    assert np.array_equal(btl, e_btl)
    assert np.array_equal(cu, np.concatenate([[0], np.cumsum(e_sq)]))


def test_effective_chunk_size():
    assert oracle.effective_chunk_size(8192, 100000, 64) == 8192
    assert oracle.effective_chunk_size(8192, 1000, 64) == 960  # min, floored to a page
    assert oracle.effective_chunk_size(8192, 10, 64) == 64  # at least one page
    assert oracle.effective_chunk_size(100, 1000, 64) == 64
