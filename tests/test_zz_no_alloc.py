"""nsa_sparse_mla_noalloc through the C ABI (GPU only).

Some callers cannot allocate device memory when they call in (a plug-in
inside a host framework that owns all device memory, a serving loop that
forbids allocation after start-up).  For them the library offers
nsa_sparse_mla_noalloc, which keeps its split-KV scratch in one fixed device
array of the library instead of a caller workspace.  The test runs two
different problems in a row through it, the larger first so that the second
call finds the first call's partials in the shared scratch, and checks each
result bit for bit against nsa_sparse_mla with a caller workspace (both run
the same kernels with the same split plan).  The file is named to run last.
"""
import ctypes as C

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _problem(seq_lens, seed):
    from deepseek_sparse_mla_indexer_gb300.step import SparseAttentionStep
    wl = W.make_workload("noalloc", mode=W.MODE_DECODE, seq_lens=seq_lens, topk=2048, page_size=64, Hi=64, Di=128,
                         idx_dtype=W.DT_E4M3, H=128, d_latent=512, d_rope=64, q_dtype=W.DT_BF16,
                         kv_dtype=W.DT_BF16, sm_scale=W.SM_SCALE_V32, seed=seed)
    st = SparseAttentionStep(wl, "cuda")
    assert st.workspace is not None, "the test problem must need scratch"
    st.metadata()
    st.indexer()
    st.topk_transform()
    st.attention()  # reference: the entry point with a caller workspace
    torch.cuda.synchronize()
    return wl, st, st.out.clone(), st.lse.clone()


def test_noalloc_matches_workspace_entry_point_bit_exact_on_two_problems():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_sparse_mla_indexer_gb300 as nsa

    lib = nsa.load()
    fn = lib.nsa_sparse_mla_noalloc
    P, I, L, F = C.c_void_p, C.c_int, C.c_int64, C.c_float
    fn.argtypes = [I, I, P, L, L, P, L, L, P, L, P, L, I, I, I, I, I, F, P, P, P, P]
    fn.restype = I
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)

    big = _problem([2500, 3100, 4000, 2049, 6000, 3333, 2100, 5000, 4500, 2600, 3900, 7000], seed=32)
    small = _problem([2500, 3100, 4000, 2049], seed=31)
    for call, (wl, st, ref_out, ref_lse) in enumerate([big, small]):
        out = torch.full_like(st.out, float("nan"))
        lse = torch.full_like(st.lse, float("nan"))
        rc = fn(st.q_dtype, st.kv_dtype, C.c_void_p(st.q_nope.data_ptr()), st.q_nope.stride(0), st.q_nope.stride(1),
                C.c_void_p(st.q_rope.data_ptr()), st.q_rope.stride(0), st.q_rope.stride(1),
                C.c_void_p(st.kv.data_ptr()), st.num_slots, C.c_void_p(st.indices.data_ptr()),
                st.indices.stride(0), wl.R, st.H, st.d_latent, st.d_rope, wl.topk, float(wl.sm_scale),
                C.c_void_p(out.data_ptr()), C.c_void_p(lse.data_ptr()), C.c_void_p(st.status.data_ptr()), stream)
        assert rc == 0, f"call {call}: {nsa.nsa_status_string(rc)}"
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}: out differs"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs"
        assert st.status_code() == 0
