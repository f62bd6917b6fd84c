"""Chunk-local dense attention on the GPU vs the oracle, through the C ABI.

The CUDA side builds its virtual batches with the library's host call
(nsa_local_virtual_batches) and runs nsa_local_attention; the oracle builds
them with its own implementation and computes the attention in float64.
out within 2e-2 * (1 + |o|) and lse within 2e-2 * (1 + |lse|) (bf16 q, K, V and
out; P rounded to bf16 for the P.V product); a row that sees no key gives out 0
and lse -inf on both sides."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import _harness as H

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_sparse_mla_indexer_gb300 as nsa
    nsa.load()


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def _gpu(q, kc, vc, bt, cu, sk, scale, q_pad=0, status=None):
    """Run nsa_local_attention on numpy inputs; returns (out float64, lse float64)."""
    import deepseek_sparse_mla_indexer_gb300 as nsa
    total, Hq, D = q.shape
    qd = torch.zeros((total, Hq * D + q_pad), dtype=torch.int16, device="cuda")
    qd[:, : Hq * D] = _dev(q.reshape(total, Hq * D), torch.int16)
    qv = qd.view(torch.bfloat16)[:, : Hq * D].view(total, Hq, D)
    out = torch.full((total, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((total, Hq), float("nan"), dtype=torch.float32, device="cuda")
    nsa.nsa_local_attention(qv, _dev(kc, torch.bfloat16), _dev(vc, torch.bfloat16), _dev(bt), _dev(cu), _dev(sk),
                            scale, out, lse, status=status)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def _through_virtual_batches(wl, rows=None):
    """GPU and oracle results of the whole local path; `rows` restricts the
    oracle to those virtual batches (the GPU always runs all of them)."""
    import deepseek_sparse_mla_indexer_gb300 as nsa
    _, cu_g, sk_g, _, bt_g = nsa.nsa_local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                           wl.block_table)
    _, cu_o, sk_o, _, bt_o = oracle.local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                          wl.block_table)
    out_g, lse_g = _gpu(wl.q, wl.k_cache, wl.v_cache, bt_g, cu_g, sk_g, wl.sm_scale)
    if rows is None:
        out_o, lse_o = oracle.local_attention(wl.q, wl.k_cache, wl.v_cache, bt_o, cu_o, sk_o, wl.sm_scale)
        return out_g, lse_g, out_o, lse_o
    # oracle on the chosen virtual batches only: their query rows, tables and key counts
    sel_q = np.concatenate([np.arange(cu_o[v], cu_o[v + 1]) for v in rows])
    cu_s = np.zeros(len(rows) + 1, np.int32)
    cu_s[1:] = np.cumsum([cu_o[v + 1] - cu_o[v] for v in rows])
    out_o, lse_o = oracle.local_attention(wl.q[sel_q], wl.k_cache, wl.v_cache, bt_o[rows], cu_s, sk_o[rows],
                                          wl.sm_scale)
    return out_g[sel_q], lse_g[sel_q], out_o, lse_o


@pytest.mark.parametrize("Hq,Hkv,D,ps,chunk", [
    (40, 8, 128, 64, 512),    # G = 5
    (32, 32, 64, 16, 256),    # G = 1
    (64, 4, 128, 16, 128),    # G = 16
    (6, 2, 64, 1, 40),        # G = 3, one token per page
])
def test_decode_through_virtual_batches(Hq, Hkv, D, ps, chunk):
    rng = np.random.default_rng(Hq * 7 + D)
    B = 7
    L = rng.integers(1, 3 * chunk + 1, size=B)
    L[0], L[1] = chunk, chunk + 1       # a full chunk, then one key into the next
    wl = W.make_local_attention("decode", seq_lens=L, q_lens=np.ones(B, np.int32), chunk=chunk, Hq=Hq, Hkv=Hkv,
                                D=D, page_size=ps, seed=int(L.sum()))
    H.check_attention(*_through_virtual_batches(wl), TOL)


@pytest.mark.parametrize("seed", [0, 1])
def test_prefill_and_extend_through_virtual_batches(seed):
    # whole prompts and partial extends that cross chunk boundaries: many
    # virtual batches with several causal query rows each
    rng = np.random.default_rng(100 + seed)
    B = 4
    L = rng.integers(40, 700, size=B)
    qn = np.array([L[0], max(1, L[1] // 3), 1, L[3] - 5], np.int32)
    wl = W.make_local_attention("prefill", seq_lens=L, q_lens=qn, chunk=128, Hq=16, Hkv=4, D=128, page_size=16,
                                seed=seed)
    H.check_attention(*_through_virtual_batches(wl), TOL)


def test_edge_batches_direct():
    # hand-made virtual batches: no keys; fewer keys than queries (leading rows
    # see nothing); exactly one tile; one key past a tile; a single key;
    # q rows with a stride larger than Hq * D
    rng = np.random.default_rng(7)
    Hq, Hkv, D, ps = 8, 2, 128, 16
    sk = np.array([0, 3, 16, 17, 1, 250], np.int32)
    nq = np.array([1, 5, 16, 2, 1, 3], np.int32)
    cu = np.zeros(len(sk) + 1, np.int32)
    cu[1:] = np.cumsum(nq)
    pages = 100
    bt = rng.permutation(pages)[: len(sk) * 16].reshape(len(sk), 16).astype(np.int32)
    kc = W._to_bf16(rng.standard_normal((pages, ps, Hkv, D)).astype(np.float32))
    vc = W._to_bf16(rng.standard_normal((pages, ps, Hkv, D)).astype(np.float32))
    q = W._to_bf16(rng.standard_normal((int(cu[-1]), Hq, D)).astype(np.float32) * 3)
    out_o, lse_o = oracle.local_attention(q, kc, vc, bt, cu, sk, 0.1)
    out_g, lse_g = _gpu(q, kc, vc, bt, cu, sk, 0.1, q_pad=24)
    H.check_attention(out_g, lse_g, out_o, lse_o, TOL)
    assert not out_g[0].any() and np.all(np.isneginf(lse_g[0]))      # batch 0 sees nothing
    assert not out_g[1:3].any() and np.all(np.isneginf(lse_g[1:3]))  # first two rows of batch 1


def test_large_logits_lazy_rescale():
    # scores that grow along the keys force the running max to move many times
    rng = np.random.default_rng(8)
    Hq, Hkv, D, ps = 4, 1, 64, 16
    n = 600
    pages = n // ps + 2
    k = rng.standard_normal((pages * ps, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    k += (np.linspace(0, 6, pages * ps)[:, None, None] * q[0, 0][None, None, :] / np.linalg.norm(q[0, 0]))
    kc = W._to_bf16(k.reshape(pages, ps, Hkv, D))
    vc = W._to_bf16(rng.standard_normal((pages, ps, Hkv, D)).astype(np.float32))
    qb = W._to_bf16(q * 4)
    bt = np.arange(pages, dtype=np.int32)[None, :]
    cu = np.array([0, 1], np.int32)
    sk = np.array([n], np.int32)
    out_o, lse_o = oracle.local_attention(qb, kc, vc, bt, cu, sk, 1.0)
    out_g, lse_g = _gpu(qb, kc, vc, bt, cu, sk, 1.0)
    H.check_attention(out_g, lse_g, out_o, lse_o, TOL)


def test_full_size_decode_sampled_rows():
    # the 32-request decode workload (chunk 8192, 40 x 8 heads, D 128) in the
    # launch the benchmark times; the oracle on 8 virtual batches incl. the longest
    wl = W.local_config("local_decode_c8192")
    _, _, sk, _, _ = oracle.local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                  wl.block_table)
    rng = np.random.default_rng(9)
    rows = sorted(set([int(np.argmax(sk)), int(np.argmin(sk)), 0, len(sk) - 1] +
                      [int(x) for x in rng.choice(len(sk), 4, replace=False)]))
    H.check_attention(*_through_virtual_batches(wl, rows), TOL)


def test_bad_page_sets_bounds():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(10)
    Hq, Hkv, D, ps = 8, 8, 64, 16
    kc = W._to_bf16(rng.standard_normal((4, ps, Hkv, D)).astype(np.float32))
    q = W._to_bf16(rng.standard_normal((1, Hq, D)).astype(np.float32))
    bt = np.array([[0, 1, 4]], np.int32)  # page 4 of a 4-page cache
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _gpu(q, kc, kc, bt, np.array([0, 1], np.int32), np.array([40], np.int32), 0.1, status=status)
    assert status.item() == nsa.ERR_BOUNDS


def test_host_rejects_bad_arguments():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    d = "cuda"
    kc = torch.zeros((2, 16, 2, 128), dtype=torch.bfloat16, device=d)
    bt = torch.zeros((1, 2), dtype=torch.int32, device=d)
    cu = torch.tensor([0, 1], dtype=torch.int32, device=d)
    sk = torch.tensor([5], dtype=torch.int32, device=d)

    def call(q, k, out, lse):
        nsa.nsa_local_attention(q, k, k, bt, cu, sk, 0.1, out, lse)

    q = torch.zeros((1, 6, 128), dtype=torch.bfloat16, device=d)
    out = torch.zeros((1, 6, 128), dtype=torch.bfloat16, device=d)
    lse = torch.zeros((1, 6), dtype=torch.float32, device=d)
    call(q, kc, out, lse)  # G = 3 is fine
    with pytest.raises(nsa.NsaError):  # Hq not a multiple of Hkv
        call(torch.zeros((1, 5, 128), dtype=torch.bfloat16, device=d), kc,
             torch.zeros((1, 5, 128), dtype=torch.bfloat16, device=d), torch.zeros((1, 5), device=d))
    with pytest.raises(nsa.NsaError):  # D = 96
        k96 = torch.zeros((2, 16, 2, 96), dtype=torch.bfloat16, device=d)
        call(torch.zeros((1, 6, 96), dtype=torch.bfloat16, device=d), k96,
             torch.zeros((1, 6, 96), dtype=torch.bfloat16, device=d), lse)
    with pytest.raises(nsa.NsaError):  # K cache not 16-byte aligned
        raw = torch.zeros(2 * 16 * 2 * 128 + 8, dtype=torch.bfloat16, device=d)
        call(q, raw[1:1 + 2 * 16 * 2 * 128].view(2, 16, 2, 128), out, lse)
    with pytest.raises(nsa.NsaError):  # G = 32 > 16
        k1 = torch.zeros((2, 16, 1, 64), dtype=torch.bfloat16, device=d)
        call(torch.zeros((1, 32, 64), dtype=torch.bfloat16, device=d), k1,
             torch.zeros((1, 32, 64), dtype=torch.bfloat16, device=d), torch.zeros((1, 32), device=d))
    # no query rows: nothing to launch
    nsa.nsa_local_attention(torch.zeros((0, 6, 128), dtype=torch.bfloat16, device=d), kc, kc, bt,
                            torch.zeros(1, dtype=torch.int32, device=d), sk[:0], 0.1,
                            torch.zeros((0, 6, 128), dtype=torch.bfloat16, device=d),
                            torch.zeros((0, 6), device=d))


def test_outputs_into_pinned_host_memory():
    # out / lse as pinned host tensors (the end-to-end benchmark's zero-copy result)
    # receive exactly what device buffers receive
    import deepseek_sparse_mla_indexer_gb300 as nsa
    wl = W.local_config("local_decode_c8192", scale=0.1)
    _, cu, sk, _, bt = nsa.nsa_local_virtual_batches(wl.chunk, wl.page_size, wl.cu_seqlens_q, wl.seq_lens,
                                                     wl.block_table)
    d = "cuda"
    q = _dev(wl.q, torch.bfloat16)
    kc, vc = _dev(wl.k_cache, torch.bfloat16), _dev(wl.v_cache, torch.bfloat16)
    args = (q, kc, vc, _dev(bt), _dev(cu), _dev(sk), wl.sm_scale)
    out = torch.empty((wl.total_q, wl.Hq, wl.D), dtype=torch.bfloat16, device=d)
    lse = torch.empty((wl.total_q, wl.Hq), dtype=torch.float32, device=d)
    nsa.nsa_local_attention(*args, out, lse)
    h_out = torch.full((wl.total_q, wl.Hq, wl.D), 3.0, dtype=torch.bfloat16).pin_memory()
    h_lse = torch.full((wl.total_q, wl.Hq), 3.0, dtype=torch.float32).pin_memory()
    nsa.nsa_local_attention(*args, h_out, h_lse)
    torch.cuda.synchronize()
    assert torch.equal(h_out.view(torch.int16), out.cpu().view(torch.int16))
    assert torch.equal(h_lse, lse.cpu())



def test_key_count_beyond_the_table_sets_bounds():
    # a seqused_k the block-table row cannot hold is reported and that batch gets no
    # keys (out 0, lse -inf); the other batch is unaffected
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(11)
    Hq, Hkv, D, ps = 8, 2, 64, 16
    kc = W._to_bf16(rng.standard_normal((6, ps, Hkv, D)).astype(np.float32))
    vc = W._to_bf16(rng.standard_normal((6, ps, Hkv, D)).astype(np.float32))
    q = W._to_bf16(rng.standard_normal((2, Hq, D)).astype(np.float32))
    bt = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    cu = np.array([0, 1, 2], np.int32)
    sk = np.array([40, 3 * ps + 1], np.int32)  # batch 1: one key past its 3-page row
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_g, lse_g = _gpu(q, kc, vc, bt, cu, sk, 0.1, status=status)
    assert status.item() == nsa.ERR_BOUNDS
    assert not out_g[1].any() and np.all(np.isneginf(lse_g[1]))
    out_o, lse_o = oracle.local_attention(q[:1], kc, vc, bt[:1], cu[:2], sk[:1], 0.1)
    H.check_attention(out_g[:1], lse_g[:1], out_o, lse_o, TOL)
