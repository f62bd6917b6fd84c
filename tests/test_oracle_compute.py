"""Pins of the oracle's indexer, top-k and sparse-MLA stages (CPU only).

The oracle is checked against special cases that reduce to a plain dot
product or a library routine, invariants, and brute force on tiny inputs --
chosen so that a dropped term, a wrong sign or index, a transposed operand or
a wrong row layout fails at least one of them.  Decoded input values come from
PyTorch's own dtype conversions, never from the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _dec_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _dec_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _small_indexer_case(seed, dtype=W.DT_E4M3, Hi=4, Di=32, ps=16, lens=(37, 70)):
    wl = W.make_workload("t", mode=W.MODE_DECODE, seq_lens=list(lens), topk=16, page_size=ps,
                         Hi=Hi, Di=Di, idx_dtype=dtype, H=2, d_latent=128, d_rope=16,
                         q_dtype=W.DT_F32, kv_dtype=W.DT_F32, sm_scale=0.1, seed=seed)
    md = oracle.metadata(wl.mode, wl.seq_lens, wl.req_to_token, wl.req_pool_indices, W=wl.W,
                         topk=wl.topk, page_size=ps)
    return wl, md


def _logits(wl, md, **over):
    args = dict(q_idx=wl.q_idx, weights=wl.weights, k_cache=wl.k_cache, k_scale=wl.k_scale,
                real_page_table=md["real_page_table"])
    args.update(over)
    return oracle.indexer_logits(wl.idx_dtype, args["q_idx"], args["weights"], args["k_cache"],
                                 args["k_scale"], args["real_page_table"], md["row_to_req"],
                                 md["seqlens_expanded"])


def _keys(wl, md, r):
    """Dequantised keys of row r, in token order, gathered with the page table."""
    ps = wl.page_size
    L = md["seqlens_expanded"][r]
    t = np.arange(L)
    slots = md["real_page_table"][md["row_to_req"][r], t // ps] * ps + t % ps
    kc = wl.k_cache.reshape(-1, wl.Di)
    k = _dec_e4m3(kc[slots]) if wl.idx_dtype == W.DT_E4M3 else kc[slots].astype(np.float64)
    return k * wl.k_scale.reshape(-1)[slots][:, None].astype(np.float64)


def _q(wl, r):
    return _dec_e4m3(wl.q_idx[r]) if wl.idx_dtype == W.DT_E4M3 else wl.q_idx[r].astype(np.float64)


# ------------------------------------------------------------------ indexer

def test_indexer_one_hot_weight_is_a_relu_dot_product():
    wl, md = _small_indexer_case(1)
    for h in range(wl.Hi):
        w = np.zeros_like(wl.weights)
        w[:, h] = 1.0
        lg = _logits(wl, md, weights=w)
        for r in range(wl.R):
            ref = np.maximum(_keys(wl, md, r) @ _q(wl, r)[h], 0.0)
            L = md["seqlens_expanded"][r]
            assert np.array_equal(lg[r, :L], ref.astype(np.float32))


def test_indexer_nonnegative_inputs_reduce_to_summed_query():
    # With q, k >= 0 every ReLU is the identity, and with w = 1 the score is
    # (sum_h q_h) . k: a plain matrix-vector product.
    wl, md = _small_indexer_case(2)
    wl.q_idx = wl.q_idx & np.uint8(0x7F)
    wl.k_cache = wl.k_cache & np.uint8(0x7F)
    lg = _logits(wl, md, q_idx=wl.q_idx, k_cache=wl.k_cache, weights=np.ones_like(wl.weights))
    for r in range(wl.R):
        ref = _keys(wl, md, r) @ _q(wl, r).sum(axis=0)
        L = md["seqlens_expanded"][r]
        np.testing.assert_allclose(lg[r, :L], ref, rtol=1e-6, atol=0)


def test_indexer_weight_sign_and_scale_are_exact():
    wl, md = _small_indexer_case(3)
    base = _logits(wl, md)
    neg = _logits(wl, md, weights=-wl.weights)
    dbl = _logits(wl, md, k_scale=wl.k_scale * np.float32(2.0))
    for r in range(wl.R):
        L = md["seqlens_expanded"][r]
        assert np.array_equal(neg[r, :L], -base[r, :L])
        assert np.array_equal(dbl[r, :L], 2 * base[r, :L])


def test_indexer_relu_is_applied_per_head_before_weighting():
    # One head with a negative dot contributes nothing; with the ReLU dropped
    # or applied after the head sum the score would change sign or size.
    wl, md = _small_indexer_case(4, Hi=2)
    w = np.ones_like(wl.weights)
    q = wl.q_idx.copy()
    q[:, 1, :] = q[:, 0, :] ^ np.uint8(0x80)  # head 1 = -head 0
    lg = _logits(wl, md, q_idx=q, weights=w)
    for r in range(wl.R):
        d0 = _keys(wl, md, r) @ _q(wl, r)[0]
        ref = np.abs(d0)  # relu(x) + relu(-x)
        L = md["seqlens_expanded"][r]
        np.testing.assert_allclose(lg[r, :L], ref, rtol=1e-6)


def test_indexer_page_placement_invariance():
    wl, md = _small_indexer_case(5, ps=8, lens=(29, 64, 3))
    base = _logits(wl, md)
    perm = np.random.default_rng(0).permutation(wl.num_pages)
    inv = np.argsort(perm)
    kc2 = wl.k_cache[inv]  # physical page p moves to position perm[p]
    ks2 = wl.k_scale[inv]
    rpt2 = perm[md["real_page_table"]].astype(np.int32)
    got = _logits(wl, md, k_cache=kc2, k_scale=ks2, real_page_table=rpt2)
    assert np.array_equal(np.nan_to_num(got, nan=7.0), np.nan_to_num(base, nan=7.0))


def test_indexer_float32_inputs_and_brute_force():
    wl, md = _small_indexer_case(6, dtype=W.DT_F32)
    lg = _logits(wl, md)
    for r in range(wl.R):
        K = _keys(wl, md, r)
        ref = np.maximum(K @ _q(wl, r).T, 0.0) @ wl.weights[r].astype(np.float64)
        L = md["seqlens_expanded"][r]
        np.testing.assert_allclose(lg[r, :L], ref, rtol=1e-6, atol=1e-6)


# ------------------------------------------------------------------ top-k

def _brute_topk(vals, L, k):
    order = sorted(range(L), key=lambda s: (1 if math.isnan(vals[s]) else 0,
                                            -(0.0 if math.isnan(vals[s]) else float(vals[s])), s))
    return sorted(order[:k]) if L > k else list(range(L))


@pytest.mark.parametrize("seed", range(5))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    R, Wd, k = 6, 90, 17
    lg = rng.integers(-4, 5, size=(R, Wd)).astype(np.float32)  # many ties
    lg[0, :8] = -0.0
    lg[1, 3] = np.nan
    L = rng.integers(0, Wd + 1, size=R).astype(np.int32)
    L[2], L[3] = k, k + 1
    pt = rng.integers(0, 10 ** 6, size=(R, Wd)).astype(np.int32)
    got = oracle.topk_transform(lg, L, np.arange(R, dtype=np.int32), pt, k)
    for r in range(R):
        pos = _brute_topk(lg[r], L[r], k)
        exp = np.full(k, -1, np.int32)
        exp[: len(pos)] = pt[r, pos]
        assert np.array_equal(got[r], exp)


def test_topk_invariants_on_distinct_values():
    rng = np.random.default_rng(11)
    R, Wd, k = 4, 5000, 300
    lg = rng.standard_normal((R, Wd)).astype(np.float32)
    L = np.array([5000, 4000, 301, 299], np.int32)
    ident = np.tile(np.arange(Wd, dtype=np.int32), (R, 1))  # transform = identity
    got = oracle.topk_transform(lg, L, np.arange(R, dtype=np.int32), ident, k)
    for r in range(R):
        n = min(L[r], k)
        sel = got[r, :n]
        assert np.all(got[r, n:] == -1)
        assert np.all(np.diff(sel) > 0) and sel.min() >= 0 and sel.max() < L[r]
        if L[r] > k:
            rest = np.setdiff1d(np.arange(L[r]), sel)
            assert lg[r, sel].min() >= lg[r, rest].max()


def test_topk_transform_uses_the_row_request_table():
    lg = np.array([[3, 1, 2, 0], [0, 1, 2, 3]], np.float32)
    pt = np.array([[10, 11, 12, 13], [20, 21, 22, 23]], np.int32)
    got = oracle.topk_transform(lg, np.array([4, 4], np.int32), np.array([1, 0], np.int32), pt, 2)
    assert np.array_equal(got, np.array([[20, 22], [12, 13]]))


def test_topk_nan_and_signed_zero():
    lg = np.array([[np.nan, -0.0, 0.0, -np.inf, np.nan]], np.float32)
    ident = np.arange(5, dtype=np.int32)[None]
    got = oracle.topk_transform(lg, np.array([5], np.int32), np.zeros(1, np.int32), ident, 2)
    assert np.array_equal(got[0], [1, 2])  # -0 == +0, NaN ranks last
    got = oracle.topk_transform(lg, np.array([5], np.int32), np.zeros(1, np.int32), ident, 4)
    assert np.array_equal(got[0], [0, 1, 2, 3])  # -inf beats NaN; lower NaN index first


# ------------------------------------------------------------------ sparse MLA

def _mla_case(seed, kv_dtype=W.DT_BF16, q_dtype=W.DT_BF16, H=4, d_latent=128, d_rope=16, lens=(50, 23)):
    wl = W.make_workload("m", mode=W.MODE_DECODE, seq_lens=list(lens), topk=64, page_size=8,
                         Hi=2, Di=16, idx_dtype=W.DT_F32, H=H, d_latent=d_latent, d_rope=d_rope,
                         q_dtype=q_dtype, kv_dtype=kv_dtype, sm_scale=(d_latent + d_rope) ** -0.5,
                         seed=seed)
    md = oracle.metadata(wl.mode, wl.seq_lens, wl.req_to_token, wl.req_pool_indices, W=wl.W,
                         topk=wl.topk, page_size=wl.page_size)
    return wl, md


def _kv_f64(wl):
    """Exact KV values [slots, d_latent + d_rope] decoded with torch."""
    if wl.kv_dtype == W.DT_F32:
        return wl.kv.astype(np.float64)
    if wl.kv_dtype == W.DT_BF16:
        return _dec_bf16(wl.kv)
    nb = wl.d_latent // 128
    lat = _dec_e4m3(wl.kv[:, : wl.d_latent]).reshape(-1, nb, 128)
    sc = np.ascontiguousarray(wl.kv[:, wl.d_latent: wl.d_latent + 4 * nb]).view(np.float32).astype(np.float64)
    rope = _dec_bf16(np.ascontiguousarray(wl.kv[:, wl.d_latent + 4 * nb:]).view(np.uint16))
    return np.concatenate([(lat * sc[:, :, None]).reshape(-1, wl.d_latent), rope], axis=1)


def _q_f64(wl, r):
    dec = _dec_bf16 if wl.q_dtype == W.DT_BF16 else (lambda a: a.astype(np.float64))
    return np.concatenate([dec(wl.q_nope[r]), dec(wl.q_rope[r])], axis=1)


@pytest.mark.parametrize("kv_dtype", [W.DT_BF16, W.DT_E4M3, W.DT_F32])
def test_sparse_equals_dense_attention_when_topk_covers_the_sequence(kv_dtype):
    # topk >= L: the sparse row selects every cached token, so sparse MLA is
    # dense single-KV-head attention (checked against torch's SDPA, fp64).
    q_dtype = W.DT_F32 if kv_dtype == W.DT_F32 else W.DT_BF16
    wl, md = _mla_case(7, kv_dtype=kv_dtype, q_dtype=q_dtype)
    idx = np.full((wl.R, wl.topk), -1, np.int32)
    for r in range(wl.R):
        L = md["seqlens_expanded"][r]
        idx[r, :L] = md["page_table_1"][r, :L]
    out, lse = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale)
    kv = _kv_f64(wl)
    for r in range(wl.R):
        L = md["seqlens_expanded"][r]
        K = torch.from_numpy(kv[md["page_table_1"][r, :L]])
        q = torch.from_numpy(_q_f64(wl, r))
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None], K[None], K[None, :, : wl.d_latent], scale=wl.sm_scale)[0]
        ref_lse = torch.logsumexp(wl.sm_scale * (q @ K.T), dim=-1)
        np.testing.assert_allclose(out[r], ref.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[r], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_single_valid_index_returns_that_value_row():
    wl, md = _mla_case(8)
    idx = np.full((wl.R, wl.topk), -1, np.int32)
    idx[:, 5] = [3, 17]
    out, lse = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale)
    kv = _kv_f64(wl)
    for r, s in enumerate([3, 17]):
        assert np.allclose(out[r], kv[s, : wl.d_latent], rtol=1e-15, atol=0)
        np.testing.assert_allclose(lse[r], wl.sm_scale * _q_f64(wl, r) @ kv[s], rtol=1e-13)


@pytest.mark.parametrize("kv_dtype", [W.DT_BF16, W.DT_E4M3])
def test_repeated_row_adds_log_count(kv_dtype):
    wl, md = _mla_case(9, kv_dtype=kv_dtype)
    n = 7
    idx = np.full((wl.R, wl.topk), -1, np.int32)
    idx[:, 10: 10 + n] = 42
    out, lse = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale)
    kv = _kv_f64(wl)
    for r in range(wl.R):
        np.testing.assert_allclose(out[r], np.broadcast_to(kv[42, : wl.d_latent], out[r].shape), rtol=1e-14)
        np.testing.assert_allclose(lse[r], wl.sm_scale * _q_f64(wl, r) @ kv[42] + math.log(n), rtol=1e-13)


def test_permutation_and_padding_invariance_and_lse_merge():
    wl, md = _mla_case(10, kv_dtype=W.DT_E4M3)
    rng = np.random.default_rng(1)
    idx = np.full((wl.R, wl.topk), -1, np.int32)
    for r in range(wl.R):
        idx[r, :40] = rng.choice(wl.num_slots, 40, replace=False)
    out, lse = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale)
    shuf = idx.copy()
    for r in range(wl.R):
        shuf[r] = shuf[r, rng.permutation(wl.topk)]
    out2, lse2 = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, shuf, wl.sm_scale)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)
    # two disjoint halves merged by their log-sum-exp give the whole
    a, b = idx.copy(), idx.copy()
    a[:, 20:] = -1
    b[:, :20] = -1
    oa, la = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, a, wl.sm_scale)
    ob, lb = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, b, wl.sm_scale)
    m = np.logaddexp(la, lb)
    np.testing.assert_allclose(m, lse, rtol=1e-13)
    merged = oa * np.exp(la - m)[..., None] + ob * np.exp(lb - m)[..., None]
    np.testing.assert_allclose(merged, out, rtol=1e-11, atol=1e-13)


def test_fp8_row_layout_latent_scale_and_rope_offsets():
    # A hand-built 656-byte row: latent code 0x38 (1.0) in block j scaled by
    # 2^j, rope bf16 0x4040 (3.0).  A one-hot query on dimension d reads back
    # exactly that element as the single score.
    d_latent, d_rope = 512, 64
    assert oracle.fp8_row_bytes(d_latent, d_rope) == 656
    row = np.zeros(656, np.uint8)
    row[:512] = 0x38
    row[512:528] = np.array([1.0, 2.0, 4.0, 8.0], np.float32).view(np.uint8)
    row[528:] = np.full(64, 0x4040, np.uint16).view(np.uint8)
    kv = np.stack([row, row])
    idx = np.array([[0, -1]], np.int32)
    for d, expect in [(0, 1.0), (130, 2.0), (300, 4.0), (511, 8.0), (512, 3.0), (575, 3.0)]:
        q = np.zeros((1, 1, 576), np.float32)
        q[0, 0, d] = 1.0
        qn = torch.from_numpy(q[..., :512]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        qr = torch.from_numpy(q[..., 512:]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        out, lse = oracle.sparse_mla(W.DT_BF16, W.DT_E4M3, qn, qr, kv, idx, 1.0)
        assert lse[0, 0] == expect
        assert np.array_equal(out[0, 0], np.repeat([1.0, 2.0, 4.0, 8.0], 128))


def test_no_valid_index_gives_zero_and_minus_inf():
    wl, md = _mla_case(12)
    idx = np.full((wl.R, wl.topk), -1, np.int32)
    out, lse = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_out_of_range_index_is_rejected():
    wl, md = _mla_case(13)
    idx = np.full((wl.R, wl.topk), -1, np.int32)
    idx[0, 0] = wl.num_slots
    with pytest.raises(ValueError):
        oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale)
