"""The C-ABI library on a machine without a GPU: it loads, exports every entry
point the header declares, and its host-side calls (local virtual batches,
effective chunk size, status strings) match the oracle and the pages'
worked example."""
import re
import os

import numpy as np
import pytest

import oracle
from tests.golden import load as load_golden

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nsa():
    import deepseek_sparse_mla_indexer_gb300 as m
    m.load()
    return m


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(nsa_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_entry_point(nsa):
    declared = _declared_functions()
    assert declared >= set(nsa.EXPORTED_SYMBOLS)
    lib = nsa.load()
    for name in sorted(declared):
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_topk_launch_plan(nsa):
    """The top-k's launch count and workspace agree: rows one CTA caches whole take
    one launch and no workspace; longer rows take per-chunk candidates plus one
    assembly, and one more launch when the indexer's digit counts are absent."""
    assert nsa.nsa_topk_launches(0, 100, False) == 0
    assert nsa.nsa_topk_launches(32, 16384, False) == 1
    assert nsa.nsa_topk_workspace_bytes(32, 16384, False) == 0
    big = 1 << 20  # rows longer than any one-CTA path
    assert nsa.nsa_topk_launches(1024, big, True) == 2
    assert nsa.nsa_topk_launches(1024, big, False) == 3
    assert nsa.nsa_topk_workspace_bytes(1024, big, False) > nsa.nsa_topk_workspace_bytes(1024, big, True) > 0


def test_status_strings(nsa):
    assert nsa.nsa_status_string(0) == "ok"
    assert "out of range" in nsa.nsa_status_string(4)
    assert nsa.nsa_abi_version() >= 100


def test_local_virtual_batches_worked_example(nsa):
    g = load_golden("local_virtual_batches_worked_example.txt")
    bt = g["block_table"].reshape(int(g["block_table_rows"][0]), int(g["block_table_cols"][0]))
    sq, cu, sk, st, btl = nsa.nsa_local_virtual_batches(int(g["attn_chunk_size"][0]), int(g["page_size"][0]),
                                                        g["query_start_loc"], g["seq_lens"], bt)
    assert np.array_equal(sq, g["seqlens_q_local"])
    assert np.array_equal(cu, g["cu_seqlens_q_local"])
    assert np.array_equal(sk, g["seqlens_k_local"])
    assert np.array_equal(st, g["k_seqstarts_absolute"])
    assert np.array_equal(btl.reshape(-1), g["block_table_local"])


@pytest.mark.parametrize("seed", range(20))
def test_local_virtual_batches_match_oracle(nsa, seed):
    rng = np.random.default_rng(1000 + seed)
    ps = int(rng.choice([1, 2, 16, 64]))
    c = ps * int(rng.integers(1, 6))
    B = int(rng.integers(1, 9))
    kv = rng.integers(1, 600, size=B)
    q = np.array([int(rng.integers(1, k + 1)) for k in kv])
    cq = np.concatenate([[0], np.cumsum(q)])
    cols = (int(kv.max()) + c) // ps + 2
    bt = rng.integers(0, 10 ** 6, size=(B, cols)).astype(np.int32)
    got = nsa.nsa_local_virtual_batches(c, ps, cq, kv, bt)
    exp = oracle.local_virtual_batches(c, ps, cq, kv, bt)
    for a, b in zip(got, exp):
        assert np.array_equal(a, b)


def test_local_virtual_batches_rejects_chunk_not_multiple_of_page(nsa):
    with pytest.raises(nsa.NsaError):
        nsa.nsa_local_virtual_batches(6, 4, np.array([0, 3]), np.array([5]), np.zeros((1, 8), np.int32))


def test_effective_chunk_size_matches_oracle(nsa):
    for c, m, ps in [(8192, 100000, 64), (8192, 1000, 64), (8192, 10, 64), (100, 1000, 64), (4, 17, 2)]:
        assert nsa.nsa_effective_chunk_size(c, m, ps) == oracle.effective_chunk_size(c, m, ps)


def _la_call(lib, **kw):
    """nsa_local_attention with fake (never dereferenced) device addresses: only the
    host-side checks run, which return before anything touches CUDA."""
    import ctypes as C
    a = dict(q=0x10000, q_ld=8 * 128, k=0x20000, v=0x30000, num_pages=4, ps=16, bt=0x40000, bt_ld=2,
             cu=0x50000, sk=0x60000, nvb=1, total_q=1, Hq=8, Hkv=2, D=128, scale=0.1, out=0x70000,
             lse=0x80000)
    a.update(kw)
    P = lambda x: C.c_void_p(x) if x else None
    return lib.nsa_local_attention(P(a["q"]), a["q_ld"], P(a["k"]), P(a["v"]), a["num_pages"], a["ps"], P(a["bt"]),
                                   a["bt_ld"], P(a["cu"]), P(a["sk"]), a["nvb"], a["total_q"], a["Hq"], a["Hkv"],
                                   a["D"], C.c_float(a["scale"]), P(a["out"]), P(a["lse"]), None, None)


def test_local_attention_host_checks(nsa):
    lib = nsa.load()
    ok, inval, unsup = 0, nsa.ERR_INVALID_ARG, nsa.ERR_UNSUPPORTED
    assert _la_call(lib, total_q=0) == ok                       # nothing to do: no launch
    assert _la_call(lib, Hq=6, Hkv=4) == inval                  # Hq not a multiple of Hkv
    assert _la_call(lib, D=96, q_ld=8 * 96) == unsup            # only D 64 and 128
    assert _la_call(lib, Hq=32, Hkv=1, q_ld=32 * 128) == unsup  # more than 16 query heads per KV head
    assert _la_call(lib, q_ld=8 * 128 - 2) == inval             # rows shorter than Hq * D
    assert _la_call(lib, q_ld=8 * 128 + 1) == inval             # odd row stride (bf16 pairs)
    assert _la_call(lib, num_pages=0) == inval                  # no page to read
    assert _la_call(lib, k=0x20008) == inval                    # K cache not 16-byte aligned
    assert _la_call(lib, q=0x10002) == inval                    # q not 4-byte aligned
    assert _la_call(lib, scale=0.0) == inval                    # sm_scale must be positive and finite
    assert _la_call(lib, scale=float("inf")) == inval
    assert _la_call(lib, lse=0) == inval                        # NULL output
    assert _la_call(lib, ps=0) == inval


def test_optional_page_table_argument_checks(nsa):
    """Host-side checks, before any launch (so they run without a device; the pointers
    are never dereferenced): nsa_metadata accepts a NULL page_table_1 but not a NULL
    real_page_table; nsa_topk_transform's row map needs a table and a row limit."""
    import ctypes as C
    lib = nsa.load()
    fake = C.c_void_p(0x1000)
    B, R, W, ps = 2, 2, 128, 64
    def md_call(pt1, real):
        o = nsa._MetadataOut(*([fake] * 8), pt1, W if pt1 else 0, real, (W + ps - 1) // ps, None, None, None)
        return lib.nsa_metadata(nsa.MODE_DECODE, B, R, W, 0, 64, ps, fake, None, fake, W, 4, fake,
                                C.byref(o), None, None)
    assert md_call(None, None) == nsa.ERR_INVALID_ARG          # no page ids buffer
    assert md_call(fake, fake) != nsa.ERR_INVALID_ARG          # passes the checks (the launch needs a device)
    assert md_call(None, fake) != nsa.ERR_INVALID_ARG          # page_table_1 may be left out
    def topk_call(pt, pt_rows, limit):
        return lib.nsa_topk_transform(fake, W, fake, fake, pt, W, pt_rows, limit, R, 64, W, fake, 64,
                                      None, None, 0, None, None)
    assert topk_call(fake, fake, 0) == nsa.ERR_INVALID_ARG     # a row map needs its row limit
    assert topk_call(None, fake, 4) == nsa.ERR_INVALID_ARG     # and a table
    assert topk_call(fake, None, 0) != nsa.ERR_INVALID_ARG
    assert topk_call(fake, fake, 4) != nsa.ERR_INVALID_ARG


def test_leading_dimension_of_one_row_views(nsa):
    import torch
    from deepseek_sparse_mla_indexer_gb300 import _ld
    assert _ld(torch.zeros(3, 5)) == 5
    assert _ld(torch.zeros(3, 8)[:, :5]) == 8           # a column slice keeps the row stride
    assert _ld(torch.zeros(5).expand(1, 5)) == 5        # broadcast row: stride 0, length 5
    assert _ld(torch.arange(5)[None, :]) == 5
    assert _ld(torch.zeros(1, 8)[:, :5]) == 5           # one row: only its length matters


@pytest.mark.parametrize("seed", range(8))
def test_local_virtual_batches_product_against_brute_force(nsa, seed):
    """The library's host builder checked directly against grouping every query
    token by the attention chunk of its own position (not against the oracle's
    restatement of the same algorithm)."""
    from tests.test_oracle_formats_metadata import _brute_force_local
    rng = np.random.default_rng(100 + seed)
    ps = int(rng.choice([1, 2, 4, 16]))
    c = ps * int(rng.integers(1, 5))
    B = int(rng.integers(1, 7))
    kv = rng.integers(1, 60, size=B)
    q = np.array([int(rng.integers(1, k + 1)) for k in kv])
    cq = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
    cols = (int(kv.max()) + c) // ps + 2
    bt = rng.integers(0, 1000, size=(B, cols)).astype(np.int32)
    sq, cu, sk, st, btl = nsa.nsa_local_virtual_batches(c, ps, cq, kv, bt)
    e_sq, e_sk, e_st, e_btl = _brute_force_local(c, ps, q, kv, bt)
    assert np.array_equal(sq, e_sq) and np.array_equal(sk, e_sk) and np.array_equal(st, e_st)
    assert np.array_equal(btl, e_btl)
    assert np.array_equal(cu, np.concatenate([[0], np.cumsum(e_sq)]))
