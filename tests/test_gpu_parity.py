"""CUDA path vs oracle, element by element, through the C ABI (GPU only).

Small cases run every row; the five named workloads at full size are checked
on sampled rows in the same launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_sparse_mla_indexer_gb300 as nsa
    nsa.load()


def _step(wl):
    from deepseek_sparse_mla_indexer_gb300.step import SparseAttentionStep
    return SparseAttentionStep(wl, "cuda")


def _mk(name, **kw):
    base = dict(mode=W.MODE_DECODE, topk=2048, page_size=64, Hi=64, Di=128, idx_dtype=W.DT_E4M3, H=128,
                d_latent=512, d_rope=64, q_dtype=W.DT_BF16, kv_dtype=W.DT_BF16, sm_scale=W.SM_SCALE_V32,
                seed=17)
    base.update(kw)
    return W.make_workload(name, **base)


SMALL = {
    # tiny float32 decode exactly as named (topk 32 < L: the selection is exercised)
    "tiny_fp32_decode": lambda: W.config("tiny_fp32_decode"),
    # tiny with topk >= L (sparse covers the whole sequence)
    "tiny_fp32_topk_covers": lambda: W.make_workload(
        "tiny_cover", mode=W.MODE_DECODE, seq_lens=[64, 100], topk=128, page_size=16, Hi=4, Di=32,
        idx_dtype=W.DT_F32, H=4, d_latent=64, d_rope=16, q_dtype=W.DT_F32, kv_dtype=W.DT_F32,
        sm_scale=80 ** -0.5, seed=1, weight_dist="uniform"),
    # bf16 decode, ragged lengths around topk and page boundaries
    "decode_bf16_ragged": lambda: _mk("dec", seq_lens=[1, 63, 2048, 2049, 3001], seed=21),
    # fp8 KV decode, 16 heads, with outliers
    "decode_fp8kv_h16": lambda: _mk("f8", seq_lens=[64, 2100, 3000, 130], H=16, kv_dtype=W.DT_E4M3,
                                    kv_outliers=0.01, seed=22),
    # chunked extend: rows cross topk inside one request
    "extend_bf16": lambda: _mk("ext", mode=W.MODE_EXTEND, seq_lens=[2100, 300], extend_lens=[80, 20], seed=23),
    # target-verify with fp8 KV
    "verify_fp8kv": lambda: _mk("ver", mode=W.MODE_VERIFY, seq_lens=[2040, 2046, 5000], n_draft=4,
                                kv_dtype=W.DT_E4M3, seed=24),
    # e4m3 indexer with a small page size and few heads (SIMT indexer path)
    "decode_small_heads_ps16": lambda: _mk("ps16", seq_lens=[33, 700, 129], page_size=16, Hi=8, Di=32,
                                           topk=256, H=16, seed=25),
}


@pytest.mark.parametrize("case", list(SMALL))
def test_small_case_all_rows(case):
    wl = SMALL[case]()
    step = _step(wl)
    rows = None if wl.R <= 8 else H.sample_rows(wl, 8, seed=1)
    H.full_parity(step, wl, rows=rows)


@pytest.mark.parametrize("case", ["decode_bf16_ragged", "decode_fp8kv_h16", "extend_bf16", "verify_fp8kv",
                                  "decode_small_heads_ps16"])
def test_small_case_other_topk_path(case):
    """The top-k path these rows (all within one CTA's reach) do not take by
    default: the indexer counting the digits for the top-k; and the metadata's
    copied page_table_1, from which the top-k then reads the slots."""
    from deepseek_sparse_mla_indexer_gb300.step import SparseAttentionStep
    wl = SMALL[case]()
    step = SparseAttentionStep(wl, "cuda", fuse_topk=True, page_table_1=True)
    rows = None if wl.R <= 8 else H.sample_rows(wl, 8, seed=3)
    H.full_parity(step, wl, rows=rows)


@pytest.mark.parametrize("name,nrows", [("v32_decode_bf16", 8), ("fp8kv_decode_h16", 6),
                                        ("chunked_extend", 4), ("verify_long_fp8kv", 4)])
def test_named_workload_full_size_sampled(name, nrows):
    """Every stage on sampled rows (the first and last rows among them; each row
    covers all its heads and every split of its top-k list), and the end-to-end
    top-k (GPU indices == the exact top-k of the GPU logits) on every row."""
    wl = W.config(name)
    step = _step(wl)
    H.full_parity(step, wl, rows=H.sample_rows(wl, nrows, seed=2), e2e_topk_rows=list(range(wl.R)))


def test_empty_batch_is_a_no_op():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    d = "cuda"
    md = nsa.alloc_metadata(nsa.MODE_DECODE, 0, 0, 0, 64, d)
    z = torch.zeros(0, dtype=torch.int32, device=d)
    r2t = torch.zeros((1, 64), dtype=torch.int32, device=d)
    nsa.nsa_metadata(nsa.MODE_DECODE, 0, 0, 0, 0, 2048, 64, z, None, r2t, z, md)
    logits = torch.zeros((0, 64), device=d)
    idx = torch.zeros((0, 2048), dtype=torch.int32, device=d)
    nsa.nsa_topk_transform(logits, z, z, md["page_table_1"], 2048, 0, idx)
    torch.cuda.synchronize()
    assert int(md["cu_seqlens_k"][0]) == 0 and int(md["nsa_cu_seqlens_k"][0]) == 0


@pytest.mark.parametrize("Wd", [40000, 70000])  # one block per row; a cluster per row
def test_topk_ties_nan_and_signed_zero_bit_exact(Wd):
    import deepseek_sparse_mla_indexer_gb300 as nsa
    import oracle
    rng = np.random.default_rng(5)
    R, k = 6, 2048
    lg = rng.integers(-3, 4, size=(R, Wd)).astype(np.float32)  # massive ties
    lg[1] = rng.standard_normal(Wd).astype(np.float32)
    lg[1, ::7] = -0.0
    lg[1, 5::11] = 0.0
    lg[2, ::3] = np.nan
    lg[3] = 1.0  # all equal: the first k positions win
    L = np.array([Wd, Wd * 6 // 7, Wd * 5 // 7 + 1, 2049, 2048, 4000], np.int32)
    pt = rng.integers(0, 2 ** 31 - 1, size=(R, Wd)).astype(np.int32)
    r2q = np.arange(R, dtype=np.int32)
    exp = oracle.topk_transform(lg, L, r2q, pt, k)
    d = "cuda"
    idx = torch.empty((R, k), dtype=torch.int32, device=d)
    nsa.nsa_topk_transform(torch.from_numpy(lg).to(d), torch.from_numpy(L).to(d), torch.from_numpy(r2q).to(d),
                           torch.from_numpy(pt).to(d), k, Wd, idx)
    assert np.array_equal(idx.cpu().numpy(), exp)


@pytest.mark.parametrize("case", ["decode_bf16_ragged", "decode_fp8kv_h16"])
def test_attention_writes_into_pinned_host_memory(case):
    # out / lse given as pinned host tensors (the end-to-end benchmark's zero-copy
    # result) receive exactly what the device buffers receive, on the in-cluster
    # merge and the combine-kernel split paths alike
    wl = SMALL[case]()
    step = _step(wl)
    step.run()
    torch.cuda.synchronize()
    h_out = torch.full(tuple(step.out.shape), 7, dtype=step.out.dtype).pin_memory()
    h_lse = torch.full(tuple(step.lse.shape), 7.0, dtype=torch.float32).pin_memory()
    step.attention(out=h_out, lse=h_lse)
    torch.cuda.synchronize()
    assert step.status_code() == 0
    assert torch.equal(h_out.view(torch.int16), step.out.cpu().view(torch.int16))
    assert torch.equal(h_lse, step.lse.cpu())


def test_out_of_range_index_sets_bounds_status():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    wl = SMALL["decode_fp8kv_h16"]()
    step = _step(wl)
    idx = torch.full((wl.R, wl.topk), -1, dtype=torch.int32, device="cuda")
    idx[:, 0] = 5
    idx[0, 1] = step.num_slots  # one past the end
    step.status.zero_()
    step.attention(indices=idx)
    assert step.status_code() == nsa.ERR_BOUNDS
    assert torch.isfinite(step.lse).all()


def test_topk_row_map_outside_the_table_sets_bounds_status():
    """A request whose row map names no row of req_to_token gets -1 slots and
    NSA_ERR_BOUNDS; the other requests' rows are unaffected."""
    import deepseek_sparse_mla_indexer_gb300 as nsa
    wl = SMALL["decode_bf16_ragged"]()
    step = _step(wl)
    step.metadata()
    step.indexer()
    step.topk_transform()
    torch.cuda.synchronize()
    good = step.indices.cpu().numpy().copy()
    assert step.status_code() == 0
    rows_map = step.md["req_rows"].clone()
    rows_map[1] = step.req_to_token.shape[0] + 5  # past the pool
    step.status.zero_()
    nsa.nsa_topk_transform(step.logits, step.md["seqlens_expanded"], step.md["row_to_req"], step.req_to_token,
                           wl.topk, wl.W, step.indices, step.status, pt_rows=rows_map)
    torch.cuda.synchronize()
    assert step.status_code() == nsa.ERR_BOUNDS
    got = step.indices.cpu().numpy()
    r2q = step.md["row_to_req"].cpu().numpy()
    for r in range(wl.R):
        if r2q[r] == 1:
            assert (got[r] == -1).all()
        else:
            assert np.array_equal(got[r], good[r])


def test_host_rejects_bad_arguments_without_launch():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    wl = SMALL["tiny_fp32_decode"]()
    step = _step(wl)
    with pytest.raises(nsa.NsaError) as e:
        nsa.nsa_topk_transform(step.logits, step.md["seqlens_expanded"], step.md["row_to_req"],
                               step.req_to_token, 0, wl.W, step.indices, pt_rows=step.md["req_rows"])
    assert e.value.code == nsa.ERR_INVALID_ARG
    with pytest.raises(nsa.NsaError) as e:  # f32 query with bf16 KV is not a supported pair
        nsa.nsa_sparse_mla(nsa.DT_F32, nsa.DT_BF16, step.q_nope, step.q_rope, step.kv, step.indices,
                           1.0, step.out, step.lse)
    assert e.value.code == nsa.ERR_UNSUPPORTED


@pytest.mark.parametrize("width", [2049, 4097, 9000, 20000, 33000, 131076])
def test_topk_bit_exact_across_row_lengths(width):
    """Rows of many lengths (short rows, one block per row; long rows, a cluster
    of blocks per row), distinct and tied scores, against the oracle."""
    import deepseek_sparse_mla_indexer_gb300 as nsa
    import oracle
    rng = np.random.default_rng(width)
    R, k = 7, 2048
    lg = rng.standard_normal((R, width)).astype(np.float32)
    lg[1] = np.round(lg[1] * 2) / 2  # coarse values: many ties across slices
    lg[2, : width // 3] = 5.0        # a plateau of equal maxima
    L = np.array([width, width - 1, width, k + 1, k, 1, max(1, width // 2)], np.int32)
    pt = rng.integers(0, 2 ** 31 - 1, size=(R, width)).astype(np.int32)
    r2q = np.arange(R, dtype=np.int32)
    exp = oracle.topk_transform(lg, L, r2q, pt, k)
    d = "cuda"
    idx = torch.empty((R, k), dtype=torch.int32, device=d)
    nsa.nsa_topk_transform(torch.from_numpy(lg).to(d), torch.from_numpy(L).to(d), torch.from_numpy(r2q).to(d),
                           torch.from_numpy(pt).to(d), k, width, idx)
    assert np.array_equal(idx.cpu().numpy(), exp)


def test_bounded_wait_times_out_and_the_context_stays_usable():
    # the wait helper of every tensor-core kernel, on a barrier nothing arrives on
    import deepseek_sparse_mla_indexer_gb300 as nsa
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nsa.nsa_check_bounded_wait(status, 100000)  # ~50 us of SM clocks
    torch.cuda.synchronize()
    assert status.item() == nsa.ERR_TIMEOUT
    # the context still runs work
    wl = SMALL["decode_small_heads_ps16"]()
    H.full_parity(_step(wl), wl)
