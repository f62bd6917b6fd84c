"""The benchmark's work accounting (CPU only): the visible-key count behind the
chunk-local attention roofline, checked against a brute-force count of the
keys each query row attends to in the oracle's virtual batches, and the
algorithmic bytes built from it."""
import numpy as np
import pytest

import bench
import oracle
import workloads as W


def _brute_visible(cu, sk):
    total = 0
    for v in range(len(sk)):
        nq, nk = int(cu[v + 1] - cu[v]), int(sk[v])
        for i in range(nq):
            total += sum(1 for j in range(nk) if j <= nk - nq + i)
    return total


@pytest.mark.parametrize("seed", range(3))
def test_visible_keys_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    B = 5
    L = rng.integers(1, 300, size=B)
    qn = np.array([int(rng.integers(1, l + 1)) for l in L], np.int32)
    wl = W.make_local_attention("acct", seq_lens=L, q_lens=qn, chunk=64, Hq=4, Hkv=2, D=64, page_size=16,
                                seed=seed)
    _, cu, sk, _, _ = oracle.local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                   wl.block_table)
    assert bench.local_visible_keys(cu, sk) == _brute_visible(cu, sk)
    # fewer keys than queries: leading rows see nothing
    assert bench.local_visible_keys(np.array([0, 5], np.int32), np.array([3], np.int32)) == 0 + 0 + 1 + 2 + 3


def test_local_bytes_decode_workload():
    # decode: one row per virtual batch, each sees all its keys
    wl = W.local_config("local_decode_c8192", scale=0.05)
    _, cu, sk, _, _ = oracle.local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                   wl.block_table)
    keys = int(sk.sum())
    assert bench.local_visible_keys(cu, sk) == keys
    pages = int(((sk + wl.page_size - 1) // wl.page_size).sum())
    expect = (keys * wl.Hkv * wl.D * 4 + wl.total_q * wl.Hq * (wl.D * 4 + 4) + pages * 4 + len(sk) * 8 + 4)
    assert bench.local_algorithmic_bytes(wl, cu, sk) == expect


def test_step_work_counts_shared_data_once():
    """Rows of one request share its key rows (indexer) and their selected KV rows
    (attention): the algorithmic bytes count them once, the flops per row."""
    wl = W.make_workload("acct", mode=W.MODE_VERIFY, seq_lens=[100, 300], n_draft=4, topk=64, page_size=16, Hi=4,
                         Di=32, idx_dtype=W.DT_E4M3, H=16, d_latent=512, d_rope=64, q_dtype=W.DT_BF16,
                         kv_dtype=W.DT_BF16, sm_scale=0.1, seed=3)
    md = oracle.metadata(wl.mode, wl.seq_lens, wl.req_to_token, wl.req_pool_indices, W=wl.W, topk=wl.topk,
                         page_size=wl.page_size, n_draft=wl.n_draft)
    L = md["seqlens_expanded"]
    r2q = md["row_to_req"]
    # every row of a request selects the same 64 slots
    idx = np.stack([np.arange(64, dtype=np.int32) + 1000 * int(b) for b in r2q])
    w = bench.algorithmic_work(wl, L, r2q, idx)
    longest = [int(L[r2q == b].max()) for b in range(2)]
    assert longest == [104, 304]
    k_bytes = sum(longest) * (32 + 4)
    pages = sum((x + 15) // 16 for x in longest) * 4
    assert w["indexer"]["bytes"] == k_bytes + int(L.sum()) * 4 + wl.R * 4 * (32 + 4) + pages
    assert w["indexer"]["flops"] == 2 * 4 * 32 * int(L.sum())
    assert w["sparse_mla"]["bytes"] == 2 * 64 * 1152 + wl.R * 16 * (576 + 512) * 2 + wl.R * 16 * 4 + wl.R * 64 * 4
    # without the indices every row's selection counts
    w2 = bench.algorithmic_work(wl, L, r2q)
    assert w2["sparse_mla"]["bytes"] - w["sparse_mla"]["bytes"] == (wl.R - 2) * 64 * 1152


def test_capture_hash_ignores_comments_but_not_code():
    """The measured DRAM traffic stays attached to a kernel through comment edits
    and is dropped by any change to its code."""
    src = ('// header\n__global__ void k(float *p) { /* body note */\n'
           '    p[0] = 1.f;  // trailing\n    asm volatile("add.f32 %0, %0, %0; // kept in the string" : "+f"(p[1]));\n}\n')
    same = src.replace("// header", "// a reworded header").replace("/* body note */", "/* another\n note */")
    code = src.replace("p[0] = 1.f;", "p[0] = 2.f;")
    lit = src.replace("// kept in the string", "// changed in the string")
    assert bench.code_only(src) == bench.code_only(same)
    assert bench.code_only(src) != bench.code_only(code)
    assert bench.code_only(src) != bench.code_only(lit)
