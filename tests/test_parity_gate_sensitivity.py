"""The parity gates catch plausible arithmetic mistakes (CPU only).

The GPU parity tests compare the CUDA path with the oracle at the method's
tolerances (tests/_harness.py): logits within 1e-3 relative, attention out and
lse within 2e-2 (bf16 KV) / 6e-2 (fp8 KV).  Here the side under test is the
oracle itself with one mistake planted in its arithmetic (the builds of
tests/test_oracle_mutants.py), run in a subprocess on small seeded decode cases
shaped like the named workloads (bf16 KV with 128 heads; fp8 KV with 16 heads
and 1 % outliers).  Each listed mistake must fail the same comparison function
the GPU tests apply: `check_logits` for the indexer's, `check_attention` (fed
the correct indices, so that only the attention's arithmetic differs) for the
attention's.

Not listed, because no tolerance can see them at these sizes and they are held
bit-exact elsewhere: a wrong decode of e4m3 subnormal codes inside fp8 KV rows
(values ~1e-3 of the block scale; the attention kernel decodes with the same
conversion and arithmetic as the paged KV dequantiser, whose GPU test is
bit-exact), and the NaN code (the workloads hold none; the format pins check it)."""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from functools import lru_cache

import numpy as np
import pytest

import oracle
import workloads as W
from tests import _harness as H
from tests.test_oracle_mutants import MUTANTS, ROOT, SRC, _build

CASES = {
    "bf16_h128": dict(mode=W.MODE_DECODE, seq_lens=[300, 2100, 2600], topk=2048, page_size=64, Hi=64, Di=128,
                      idx_dtype=W.DT_E4M3, H=128, d_latent=512, d_rope=64, q_dtype=W.DT_BF16,
                      kv_dtype=W.DT_BF16, sm_scale=W.SM_SCALE_V32, seed=31),
    "fp8_h16": dict(mode=W.MODE_DECODE, seq_lens=[300, 2100, 2600], topk=2048, page_size=64, Hi=64, Di=128,
                    idx_dtype=W.DT_E4M3, H=16, d_latent=512, d_rope=64, q_dtype=W.DT_BF16, kv_dtype=W.DT_E4M3,
                    kv_outliers=0.01, sm_scale=W.SM_SCALE_V32, seed=32),
}

_LOGIT_MISTAKES = ["indexer_relu_dropped", "indexer_relu_after_weight", "indexer_key_scale_dropped",
                   "indexer_slot_in_page", "e4m3_exponent_bias", "e4m3_subnormal_scale"]
_ATTN_MISTAKES = ["mla_rope_dropped", "mla_scale_dropped", "mla_lse_base_2", "mla_value_reversed"]
_FP8_ATTN_MISTAKES = ["fp8_scale_block_shifted", "fp8_rope_offset", "e4m3_exponent_bias"]

# (case, planted mistake, gate that must fail)
GATES = ([(c, m, "logits") for c in CASES for m in _LOGIT_MISTAKES] +
         [(c, m, "attention") for c in CASES for m in _ATTN_MISTAKES] +
         [("fp8_h16", m, "attention") for m in _FP8_ATTN_MISTAKES])

# Run in the subprocess with NSA_ORACLE_LIB naming the build under test.
_PROBE = r"""
import json, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import oracle, workloads as W
kw, gate, idx_path, out_path = json.loads(sys.argv[2]), sys.argv[3], sys.argv[4], sys.argv[5]
wl = W.make_workload("gate", **kw)
if gate == "logits":
    md = oracle.metadata(wl.mode, wl.seq_lens, wl.req_to_token, wl.req_pool_indices, W=wl.W, topk=wl.topk,
                         page_size=wl.page_size, extend_lens=wl.extend_lens, n_draft=wl.n_draft)
    lg = oracle.indexer_logits(wl.idx_dtype, wl.q_idx, wl.weights, wl.k_cache, wl.k_scale,
                               md["real_page_table"], md["row_to_req"], md["seqlens_expanded"])
    np.savez(out_path, lg=lg)
else:
    out, lse = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, np.load(idx_path),
                                 wl.sm_scale)
    np.savez(out_path, out=out, lse=lse)
"""

_OUT = os.path.join(ROOT, "oracle", "_build", "gate")


@lru_cache(maxsize=None)
def _reference(case):
    """The unmodified oracle's logits, indices and attention for a case (computed once)."""
    wl = W.make_workload("gate", **CASES[case])
    md = H.oracle_metadata(wl)
    lg = oracle.indexer_logits(wl.idx_dtype, wl.q_idx, wl.weights, wl.k_cache, wl.k_scale,
                               md["real_page_table"], md["row_to_req"], md["seqlens_expanded"])
    idx = oracle.topk_transform(lg, md["seqlens_expanded"], md["row_to_req"], md["page_table_1"], wl.topk)
    out, lse = oracle.sparse_mla(wl.q_dtype, wl.kv_dtype, wl.q_nope, wl.q_rope, wl.kv, idx, wl.sm_scale)
    return dict(wl=wl, lens=md["seqlens_expanded"], lg=lg, idx=idx, out=out, lse=lse)


def _gate_outcome(job):
    case, name, gate, ref, so = job
    idx_path = os.path.join(_OUT, f"{case}_idx.npy")
    out_path = os.path.join(_OUT, f"{case}_{name}_{gate}.npz")
    env = dict(os.environ, NSA_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-c", _PROBE, ROOT, json.dumps(CASES[case]), gate, idx_path, out_path],
                       env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return f"{case}/{name}: the probe failed: {r.stderr[-1500:]}"
    m = np.load(out_path)
    try:
        if gate == "logits":
            H.check_logits(m["lg"], ref["lg"], ref["lens"])
        else:
            H.check_attention(m["out"], m["lse"], ref["out"], ref["lse"], H.attn_tol(ref["wl"]))
    except AssertionError:
        return None
    return f"{case}/{name}: passed the {gate} gate"


def test_cases_exercise_the_selection():
    """Rows both shorter and longer than topk, every head with a finite lse."""
    for case in CASES:
        ref = _reference(case)
        assert (ref["lens"] < ref["wl"].topk).any() and (ref["lens"] > ref["wl"].topk).any()
        assert np.isfinite(ref["lse"]).all()


def test_every_listed_mistake_fails_its_gate():
    os.makedirs(_OUT, exist_ok=True)
    with open(SRC) as f:
        src = f.read()
    edits = {name: (old, new) for name, old, new, _ in MUTANTS}
    refs = {}
    for case in CASES:
        refs[case] = _reference(case)
        np.save(os.path.join(_OUT, f"{case}_idx.npy"), refs[case]["idx"])
    builds = {}
    for _, name, _ in GATES:
        if name not in builds:
            old, new = edits[name]
            builds[name] = _build(name, src.replace(old, new))
    jobs = [(case, name, gate, refs[case], builds[name]) for case, name, gate in GATES]
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        missed = [m for m in ex.map(_gate_outcome, jobs) if m is not None]
    assert not missed, missed


@pytest.mark.parametrize("case", list(CASES))
def test_rounding_sized_differences_pass(case):
    """The gates are not so tight that arithmetic in another order fails them:
    outputs perturbed by a relative 1e-4 (logits) / 2e-3 (attention) pass."""
    ref = _reference(case)
    rng = np.random.default_rng(5)
    lg = ref["lg"].astype(np.float64)
    lg_p = (lg * (1 + 1e-4 * rng.uniform(-1, 1, lg.shape))).astype(np.float32)
    H.check_logits(lg_p, ref["lg"], ref["lens"])
    out_p = ref["out"] * (1 + 2e-3 * rng.uniform(-1, 1, ref["out"].shape))
    lse_p = ref["lse"] * (1 + 2e-3 * rng.uniform(-1, 1, ref["lse"].shape))
    H.check_attention(out_p, lse_p, ref["out"], ref["lse"], H.attn_tol(ref["wl"]))
