"""The top-k's use of the indexer's digit counts (GPU only, through the C ABI).

nsa_topk_transform may be given the per-row counts of the scores' leading 11
key bits that nsa_indexer_logits accumulates.  The counts are only a hint: the
indices must equal the oracle's whatever the buffer holds (exact counts, zeros,
garbage, counts of other scores, counts moved between bins with the total kept),
and every row of the buffer is zero afterwards."""
import numpy as np
import pytest
import torch

from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_sparse_mla_indexer_gb300 as nsa
    nsa.load()


def _rows(width, seed):
    rng = np.random.default_rng(seed)
    R = 8
    lg = rng.standard_normal((R, width)).astype(np.float32)
    lg[1] = np.round(lg[1] * 2) / 2           # coarse values: crowded bins and ties
    lg[2, : width // 3] = 5.0                 # a plateau of equal maxima
    lg[3, ::7] = -0.0                         # signed zeros among normal scores
    lg[3, 5::11] = 0.0
    lg[4, ::3] = np.nan                       # NaN ranks lowest
    lg[5] = np.abs(lg[5]) * 1e-3 + 1.0        # a narrow band: one leading digit holds every score
    L = np.array([width, width - 1, width, max(2049, width // 2), width, width, 2048, 1], np.int32)
    return lg, L


def _hint(kind, lg, L, rng):
    exact = H.host_digit_hist(lg, L)
    if kind == "exact":
        return exact
    if kind == "zero":
        return np.zeros_like(exact)
    if kind == "garbage":
        return rng.integers(0, 1 << 20, size=exact.shape)
    if kind == "other_scores":  # the counts of different scores with the same lengths
        other = rng.standard_normal(lg.shape).astype(np.float32) * 3
        return H.host_digit_hist(other, L)
    if kind == "moved_count":  # one key moved to a neighbouring bin: the total still matches
        h = exact.copy()
        for i in range(len(L)):
            nz = np.nonzero(h[i])[0]
            if len(nz):
                d = nz[-1]  # the highest occupied bin
                h[i, d] -= 1
                h[i, d - 1 if d > 0 else d + 1] += 1
        return h
    raise KeyError(kind)


@pytest.mark.parametrize("kind", ["exact", "zero", "garbage", "other_scores", "moved_count"])
@pytest.mark.parametrize("width", [2049, 9000, 33000, 40960, 70000])
def test_topk_bit_exact_whatever_the_digit_counts(kind, width):
    import deepseek_sparse_mla_indexer_gb300 as nsa
    import oracle
    rng = np.random.default_rng(width + len(kind))
    lg, L = _rows(width, seed=width)
    k = 2048
    R = len(L)
    pt = rng.integers(0, 2 ** 31 - 1, size=(R, width)).astype(np.int32)
    r2q = np.arange(R, dtype=np.int32)
    exp = oracle.topk_transform(lg, L, r2q, pt, k)
    d = "cuda"
    hist = torch.from_numpy(_hint(kind, lg, L, rng).astype(np.uint32).view(np.int32)).to(d)
    idx = torch.empty((R, k), dtype=torch.int32, device=d)
    nsa.nsa_topk_transform(torch.from_numpy(lg).to(d), torch.from_numpy(L).to(d), torch.from_numpy(r2q).to(d),
                           torch.from_numpy(pt).to(d), k, width, idx, score_hist=hist)
    got = idx.cpu().numpy()
    bad = [i for i in range(R) if not np.array_equal(got[i], exp[i])]
    assert not bad, f"rows {bad} differ from the oracle with {kind} digit counts"
    assert not hist.any().item(), "digit counts left behind"


def test_ragged_topk_with_digit_counts():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    import oracle
    rng = np.random.default_rng(3)
    width, k = 12000, 2048
    lg, L = _rows(width, seed=3)
    R = len(L)
    r2q = (np.arange(R) % 3).astype(np.int32)
    off = np.array([0, 50000, 123457], np.int32)
    exp = oracle.topk_ragged(lg, L, r2q, off, k)
    d = "cuda"
    hist = torch.from_numpy(H.host_digit_hist(lg, L).astype(np.uint32).view(np.int32)).to(d)
    idx = torch.empty((R, k), dtype=torch.int32, device=d)
    nsa.nsa_topk_transform_ragged(torch.from_numpy(lg).to(d), torch.from_numpy(L).to(d),
                                  torch.from_numpy(r2q).to(d), torch.from_numpy(off).to(d), k, width, idx,
                                  score_hist=hist)
    assert np.array_equal(idx.cpu().numpy(), exp)
    assert not hist.any().item()


@pytest.mark.parametrize("mode", ["decode", "verify", "extend"])
def test_indexer_digit_counts_equal_those_of_its_logits(mode):
    """One row per group (decode) and four rows per group (verify, extend), rows
    longer than one flush interval of the per-CTA counters (256 tiles)."""
    import workloads as W
    from deepseek_sparse_mla_indexer_gb300.step import SparseAttentionStep
    kw = dict(topk=2048, page_size=64, Hi=64, Di=128, idx_dtype=W.DT_E4M3, H=16, d_latent=512, d_rope=64,
              q_dtype=W.DT_BF16, kv_dtype=W.DT_BF16, sm_scale=W.SM_SCALE_V32, seed=41)
    if mode == "decode":
        wl = W.make_workload("dh", mode=W.MODE_DECODE, seq_lens=[70000, 5, 2048, 33000, 129], **kw)
    elif mode == "verify":
        wl = W.make_workload("vh", mode=W.MODE_VERIFY, seq_lens=[40000, 3000], n_draft=4, **kw)
    else:
        wl = W.make_workload("eh", mode=W.MODE_EXTEND, seq_lens=[9000, 2300], extend_lens=[37, 6], **kw)
    st = SparseAttentionStep(wl, "cuda", fuse_topk=True)
    st.metadata()
    st.indexer()
    torch.cuda.synchronize()
    lens = st.md["seqlens_expanded"].cpu().numpy()
    rows = list(range(wl.R))
    H.check_digit_hist(st, rows, st.logits.cpu().numpy(), lens)
    st.topk_transform()
    torch.cuda.synchronize()
    assert not st.score_hist.any().item()
    assert st.status_code() == 0
