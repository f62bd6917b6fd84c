"""Mutation check of the oracle's pins (CPU only).

Each mutant is the oracle's C source with one plausible mistake planted in it: a
wrong exponent bias or rounding rule, a dropped term, a flipped sign or
comparison, a transposed or shifted index.  Every mutant is compiled on its own
and loaded, through `NSA_ORACLE_LIB`, by the oracle's own pin tests
(tests/test_oracle_*.py) in a subprocess; each must make at least one pin fail.
The unmodified source, built and loaded the same way, must pass them all, so a
failure is the planted mistake's and not the harness's.  The mutants change
arithmetic only, never a bound: a planted mistake reads no memory the original
does not.

Builds go to oracle/_build/mutants/<name>/ (not tracked)."""
import os
import subprocess
import sys

from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nsa_oracle.c")
OUT = os.path.join(ROOT, "oracle", "_build", "mutants")
PINS = {
    "compute": "tests/test_oracle_compute.py",
    "formats": "tests/test_oracle_formats_metadata.py",
    "kvwrite": "tests/test_oracle_kvwrite.py",
    "local": "tests/test_oracle_local_attention.py",
}
# the one slow pin (a full-size metadata call); every mutant below is caught without it
SKIP_SLOW = "not named_workload_rows"

# (name, text in the oracle source, its replacement, pin files expected to catch it)
MUTANTS = [
    # number formats
    ("e4m3_subnormal_scale", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);", ["formats"]),
    ("e4m3_exponent_bias", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);", ["formats"]),
    ("e4m3_nan_code", "if (e == 0xF && m == 0x7)", "if (e == 0xF && m == 0x8)", ["formats"]),
    ("e4m3_encode_ties_away", "double m = nearbyint((fr * 2.0 - 1.0) * 8.0);",
     "double m = floor((fr * 2.0 - 1.0) * 8.0 + 0.5);", ["kvwrite"]),
    ("e4m3_encode_subnormal_step", "double m = nearbyint(a * 512.0);", "double m = nearbyint(a * 256.0);",
     ["kvwrite"]),
    ("bf16_truncates", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;", ["kvwrite"]),
    ("block_scale_divisor", "scale = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "scale = amax > 0.0f ? amax / 240.0f : 1.0f;", ["kvwrite"]),
    ("mla_row_scale_slot", "memcpy(row + d_latent + 4 * b, &sc, 4);",
     "memcpy(row + d_latent + 4 * (d_latent / 128 - 1 - b), &sc, 4);", ["kvwrite"]),
    # metadata and local virtual batches
    ("verify_drafts_not_cached", "cache_seqlens[b] = seq_lens[b] + draft;", "cache_seqlens[b] = seq_lens[b];",
     ["formats"]),
    ("expanded_off_by_one", "seqlens_expanded[r] = kv - q + 1 + i;", "seqlens_expanded[r] = kv - q + i;",
     ["formats"]),
    ("no_topk_clip", "nsa_cache_seqlens[i] = L < topk ? L : topk;", "nsa_cache_seqlens[i] = L;", ["formats"]),
    ("page_id_not_divided", "(int32_t)py_floordiv(src[p * page_size], page_size);", "(int32_t)src[p * page_size];",
     ["formats"]),
    ("ke_off_by_one", "ke[r] = (int32_t)(k_offset + seqlens_expanded[r]);",
     "ke[r] = (int32_t)(k_offset + seqlens_expanded[r] - 1);", ["formats"]),
    ("last_block_keys_full_chunk", "sk = (j == blocks - 1) ? last : c;", "sk = c;", ["formats"]),
    ("later_block_queries_clipped_short", "if (sq > c) sq = c;", "if (sq > c) sq = c - 1;", ["formats"]),
    ("chunk_not_page_rounded", "c = (c / page_size) * page_size;", "c = c;", ["formats"]),
    # indexer
    ("indexer_relu_dropped", "acc += (double)w_row[h] * (dot > 0.0 ? dot : 0.0);", "acc += (double)w_row[h] * dot;",
     ["compute"]),
    ("indexer_relu_after_weight", "acc += (double)w_row[h] * (dot > 0.0 ? dot : 0.0);",
     "acc += ((double)w_row[h] * dot > 0.0 ? (double)w_row[h] * dot : 0.0);", ["compute"]),
    ("indexer_key_scale_dropped", "scale = (double)k_scale[slot];", "scale = 1.0;", ["compute"]),
    ("indexer_slot_in_page", "slot = page * ps + s % ps;", "slot = page * ps + (s + 1) % ps;", ["compute"]),
    # top-k and its transform
    ("topk_ties_to_higher_position", "return (a->s > b->s) - (a->s < b->s);", "return (a->s < b->s) - (a->s > b->s);",
     ["compute"]),
    ("topk_nan_on_top", "if (an != bn) return an ? 1 : -1;", "if (an != bn) return an ? -1 : 1;", ["compute"]),
    ("topk_positions_unsorted", "qsort(pos, (size_t)topk, sizeof(int32_t), orc_int_cmp);", "(void)orc_int_cmp;",
     ["compute"]),
    ("topk_pad_zero", "for (int i = n; i < topk; ++i) out_row[i] = -1;",
     "for (int i = n; i < topk; ++i) out_row[i] = 0;", ["compute"]),
    ("ragged_offset_sign", "if (out_row[i] != -1) out_row[i] += offset;", "if (out_row[i] != -1) out_row[i] -= offset;",
     ["kvwrite"]),
    ("flatten_drops_last", "for (int t = 0; t < kv_len[b]; ++t) out[n++]",
     "for (int t = 0; t < kv_len[b] - 1; ++t) out[n++]", ["kvwrite"]),
    # sparse MLA
    ("mla_rope_dropped", "for (int d = 0; d < d_rope; ++d)\n                dot += load_elem(q_rope",
     "for (int d = 0; d < 0; ++d)\n                dot += load_elem(q_rope", ["compute"]),
    ("mla_scale_dropped", "kv_elem(kv, kv_dtype, d_latent, d_rope, slot, d_latent + d);\n            s[j] = sm_scale * dot;",
     "kv_elem(kv, kv_dtype, d_latent, d_rope, slot, d_latent + d);\n            s[j] = dot;", ["compute"]),
    ("mla_lse_base_2", "l = m + log(sum);", "l = m + log2(sum);", ["compute"]),
    ("mla_value_reversed", "out[(int64_t)h * d_latent + d] += p * kv_elem(kv, kv_dtype, d_latent, d_rope, slot, d);",
     "out[(int64_t)h * d_latent + d] += p * kv_elem(kv, kv_dtype, d_latent, d_rope, slot, d_latent - 1 - d);",
     ["compute"]),
    ("fp8_scale_block_shifted", "memcpy(&sc, row + d_latent + 4 * (d / 128), 4);\n            return",
     "memcpy(&sc, row + d_latent + 4 * ((d / 128 + 1) % (d_latent / 128)), 4);\n            return", ["compute"]),
    ("fp8_rope_offset", "memcpy(&h, row + d_latent + 4 * (d_latent / 128) + 2 * (d - d_latent), 2);",
     "memcpy(&h, row + d_latent + 2 * (d - d_latent), 2);", ["compute"]),
    # chunk-local attention
    ("local_not_causal", "int last = nk - nq + i; /* last key this query sees */", "int last = nk - 1;", ["local"]),
    ("local_head_group_map", "int hk = h / G;", "int hk = h % Hkv;", ["local"]),
]


def _build(name: str, text: str) -> str:
    d = os.path.join(OUT, name)
    os.makedirs(d, exist_ok=True)
    c, so = os.path.join(d, "nsa_oracle.c"), os.path.join(d, "liboracle.so")
    with open(c, "w") as f:
        f.write(text)
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                           "-o", so, c, "-lm"])
    return so


def _run_pins(so: str, files) -> subprocess.CompletedProcess:
    env = dict(os.environ, NSA_ORACLE_LIB=so)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", "-k", SKIP_SLOW,
           *files]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unmodified_oracle_passes_its_pins_when_loaded_the_same_way():
    with open(SRC) as f:
        src = f.read()
    r = _run_pins(_build("unmodified", src), list(PINS.values()))
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_mutant_names_are_unique():
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))


def _mutant_outcome(m):
    name, old, new, pins = m
    with open(SRC) as f:
        src = f.read()
    if src.count(old) != 1:
        return name, "the text to replace does not occur exactly once"
    r = _run_pins(_build(name, src.replace(old, new)), [PINS[p] for p in pins])
    # exit status 1: the pins ran and at least one failed (not a crash, a
    # collection error or an interrupted run)
    return name, None if r.returncode == 1 else f"survived (exit {r.returncode}): {r.stdout[-1500:]}"


def test_every_planted_mistake_fails_a_pin():
    """The mutants run concurrently, each in its own process."""
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        outcomes = list(ex.map(_mutant_outcome, MUTANTS))
    survivors = {n: why for n, why in outcomes if why is not None}
    assert not survivors, survivors
