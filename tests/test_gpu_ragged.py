"""RAGGED extend on the GPU vs the oracle, through the C ABI: the ragged top-k
(positions + request offset) and the flattened page table bit-exact, and the
whole RAGGED path (flatten -> dequantise the fp8 cache into a request-contiguous
bf16 KV -> ragged top-k -> sparse MLA) against the oracle's paged attention."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_sparse_mla_indexer_gb300 as nsa
    nsa.load()


@pytest.mark.parametrize("width", [3000, 30000, 70000])  # short rows, one block per row, a cluster per row
def test_ragged_topk_bit_exact(width):
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(width)
    R, k = 9, 2048
    lg = rng.standard_normal((R, width)).astype(np.float32)
    lg[2] = np.round(lg[2] * 2) / 2  # ties
    L = np.array([width, width - 7, 2049, 2048, 1, width // 2, width, 100, width // 3], np.int32)
    r2q = np.array([0, 0, 1, 1, 2, 3, 3, 3, 4], np.int32)  # extend: several rows per request
    offsets = np.array([0, 123457, 200000, 300001, 999999], np.int32)
    exp = oracle.topk_ragged(lg, L, r2q, offsets, k)
    d = "cuda"
    idx = torch.empty((R, k), dtype=torch.int32, device=d)
    nsa.nsa_topk_transform_ragged(torch.from_numpy(lg).to(d), torch.from_numpy(L).to(d),
                                  torch.from_numpy(r2q).to(d), torch.from_numpy(offsets).to(d), k, width, idx)
    assert np.array_equal(idx.cpu().numpy(), exp)


def test_flatten_page_table_bit_exact():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(31)
    B, Wd = 7, 9000
    pt = rng.integers(0, 2 ** 31 - 1, size=(B, Wd)).astype(np.int32)
    kv = np.array([9000, 0, 4097, 1, 8191, 4096, 300], np.int32)
    start = np.concatenate([[0], np.cumsum(kv)[:-1]]).astype(np.int32)
    out = torch.full((int(kv.sum()),), -5, dtype=torch.int32, device="cuda")
    nsa.nsa_flatten_page_table(torch.from_numpy(pt).cuda(), torch.from_numpy(kv).cuda(),
                               torch.from_numpy(start).cuda(), out)
    assert np.array_equal(out.cpu().numpy(), oracle.flatten_page_table(pt, kv))


def test_ragged_extend_path_matches_paged_attention():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    from deepseek_sparse_mla_indexer_gb300.step import SparseAttentionStep
    # 18 extend rows x 64 heads (the tensor-core shapes) keep the fp64 oracle to seconds
    wl = W.make_workload("ragged", mode=W.MODE_EXTEND, seq_lens=[2100, 300, 2600], extend_lens=[8, 4, 6],
                         topk=2048, page_size=64, Hi=64, Di=128, idx_dtype=W.DT_E4M3, H=64, d_latent=512,
                         d_rope=64, q_dtype=W.DT_BF16, kv_dtype=W.DT_E4M3, sm_scale=W.SM_SCALE_V32, seed=33)
    st = SparseAttentionStep(wl, "cuda", page_table_1=True)
    st.metadata()
    torch.cuda.synchronize()
    md_o = H.oracle_metadata(wl)
    rows = list(range(wl.R))
    lg = oracle.indexer_logits(wl.idx_dtype, wl.q_idx, wl.weights, wl.k_cache, wl.k_scale, md_o["real_page_table"],
                               md_o["row_to_req"], md_o["seqlens_expanded"], rows=rows, width=wl.W)
    # request-contiguous KV: flatten the page table, gather and dequantise the fp8 rows
    kv_len, kv_start = st.md["cache_seqlens"], st.md["cu_seqlens_k"][:-1].contiguous()
    total = int(md_o["cu_seqlens_k"][-1])
    flat = torch.empty((total,), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nsa.nsa_flatten_page_table(st.md["page_table_1"], kv_len, kv_start, flat, status)
    ragged_kv = torch.empty((total, 576), dtype=torch.int16, device="cuda")
    nsa.nsa_dequantize_kv_paged(st.kv, flat, ragged_kv, status=status)
    # ragged top-k on the oracle's logits, then the attention over the ragged KV
    logits = torch.full((wl.R, st.logits.shape[1]), float("-inf"), dtype=torch.float32, device="cuda")
    logits[:, : wl.W] = torch.from_numpy(lg)
    idx = torch.empty((wl.R, wl.topk), dtype=torch.int32, device="cuda")
    nsa.nsa_topk_transform_ragged(logits, st.md["seqlens_expanded"], st.md["row_to_req"], kv_start, wl.topk,
                                  wl.W, idx, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    exp_idx = oracle.topk_ragged(lg, md_o["seqlens_expanded"], md_o["row_to_req"], md_o["cu_seqlens_k"][:-1],
                                 wl.topk)
    assert np.array_equal(idx.cpu().numpy(), exp_idx)
    out = torch.empty((wl.R, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.R, wl.H), dtype=torch.float32, device="cuda")
    ws_bytes = nsa.nsa_sparse_mla_workspace_bytes(W.DT_BF16, W.DT_BF16, wl.R, wl.H, 512, 64, wl.topk)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    nsa.nsa_sparse_mla(W.DT_BF16, W.DT_BF16, st.q_nope, st.q_rope, ragged_kv.view(torch.bfloat16), idx,
                       float(wl.sm_scale), out, lse, ws, status, num_slots=total)
    torch.cuda.synchronize()
    assert status.item() == 0
    # the oracle's attention over the paged fp8 cache with the paged indices of the same selection
    paged_idx = oracle.topk_transform(lg, md_o["seqlens_expanded"], md_o["row_to_req"], md_o["page_table_1"],
                                      wl.topk, rows=rows, logits_rows_are_subset=True)
    out_o, lse_o = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, paged_idx, wl.sm_scale,
                                     rows=rows, indices_rows_are_subset=True)
    H.check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o, H.attn_tol(wl))
