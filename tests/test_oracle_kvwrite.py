"""Pins of the oracle's KV-cache write side (CPU only): the e4m3 encoder, the
bf16 rounding, and the row quantisers behind set_mla_kv_buffer /
quantize_k_cache / dequantize_k_cache_paged and the indexer key rows.

Each check ties the oracle to something other than itself: the format's own
values, PyTorch's float8 / bfloat16 casts, the workload generator's separate
quantiser, and invariants of the rounding."""
import numpy as np
import torch

import oracle
import workloads as W


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_of(x: np.ndarray) -> np.ndarray:
    return _torch_bf16(x)


def _f32_from_bf16(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ e4m3 encode

def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_midpoints_round_to_even_and_neighbours_to_nearest():
    pos = np.arange(0x00, 0x7E, dtype=np.uint8)  # adjacent finite pairs (c, c+1)
    lo = oracle.e4m3_to_f64(pos)
    hi = oracle.e4m3_to_f64(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)  # exact in fp32
    got = oracle.e4m3_encode(mid)
    even = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(got, even)
    below = np.nextafter(mid, np.float32(-np.inf))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(oracle.e4m3_encode(below), pos)
    assert np.array_equal(oracle.e4m3_encode(above), pos + 1)
    assert np.array_equal(oracle.e4m3_encode(-mid), even | 0x80)


def test_encode_matches_torch_cast_within_range():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.uniform(-463.9, 463.9, 20000), rng.standard_normal(20000) * 0.01,
                        rng.standard_normal(20000) * 2.0 ** -8]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3(x))


def test_encode_saturates_and_keeps_nan():
    got = oracle.e4m3_encode(np.array([464.0, 500.0, 1e30, -1e30, np.nan], np.float32))
    assert list(got[:4]) == [0x7E, 0x7E, 0x7E, 0xFE]
    assert got[4] == 0x7F


def test_f32_to_bf16_matches_torch_cast():
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000),
                        [0.0, -0.0, 1.0, 65504.0, 3.4e38, -3.4e38, 1e-40]]).astype(np.float32)
    assert np.array_equal(oracle.f32_to_bf16(x), _torch_bf16(x))


# ------------------------------------------------------------------ row quantisers

def _rows(rng, n, d):
    x = rng.standard_normal((n, d)).astype(np.float32)
    x[0, :128] = 0.0                    # an all-zero block
    x[1, 5] = 37.0                      # an outlier block
    x[2, :] *= 1e-3                     # small values (subnormal codes)
    return _bf16_of(x)


def test_index_rows_match_the_generators_quantiser():
    # the workload generator quantises with numpy + torch casts, a separate code path
    rng = np.random.default_rng(13)
    k = _rows(rng, 64, 128)
    codes, scales = oracle.quantize_index_rows(k)
    exp_codes, exp_scales = W._e4m3_rows_with_scale(_f32_from_bf16(k), 128)
    assert np.array_equal(scales, exp_scales[:, 0])
    assert np.array_equal(codes, exp_codes)


def test_mla_row_layout_and_closed_forms():
    rng = np.random.default_rng(14)
    lat = _rows(rng, 16, 512)
    rope = _bf16_of(rng.standard_normal((16, 64)).astype(np.float32))
    rows = oracle.quantize_mla_rows(lat, rope)
    assert rows.shape == (16, oracle.fp8_row_bytes(512, 64)) == (16, 656)
    latf = _f32_from_bf16(lat).reshape(16, 4, 128)
    amax = np.abs(latf).max(axis=2)
    scales = rows[:, 512:528].copy().view(np.float32).reshape(16, 4)
    assert np.array_equal(scales, np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32))
    assert scales[0, 0] == 1.0 and not rows[0, :128].any()          # zero block
    # the largest magnitude of each non-zero block encodes to +-448
    codes = rows[:, :512].reshape(16, 4, 128)
    arg = np.abs(latf).argmax(axis=2)
    top = np.take_along_axis(codes, arg[..., None], axis=2)[..., 0]
    assert np.all(((top & 0x7F) == 0x7E) | (amax == 0))
    # codes agree with torch's cast of x / scale (all within the finite range)
    q = (latf / scales[..., None]).astype(np.float32)
    assert np.array_equal(codes, _torch_e4m3(q))
    # the rope part is copied bit for bit
    assert np.array_equal(rows[:, 528:].copy().view(np.uint16), rope)


def test_mla_dequantize_round_trip():
    rng = np.random.default_rng(15)
    lat = _rows(rng, 16, 512)
    rope = _bf16_of(rng.standard_normal((16, 64)).astype(np.float32))
    rows = oracle.quantize_mla_rows(lat, rope)
    back = oracle.dequantize_mla_rows(rows, 512, 64)
    assert np.array_equal(back[:, 512:], rope)
    # latent: bf16(fp32(code value x scale)) with torch's decode and casts
    scales = rows[:, 512:528].copy().view(np.float32).reshape(16, 4)
    vals = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    prod = (vals.reshape(16, 4, 128) * scales[..., None]).astype(np.float32).reshape(16, 512)
    assert np.array_equal(back[:, :512], _torch_bf16(prod))
    # quantisation error: at most half an e4m3 step of each value (relative 2^-4), plus bf16 rounding
    x = _f32_from_bf16(lat).astype(np.float64)
    y = _f32_from_bf16(back[:, :512]).astype(np.float64)
    sc = np.repeat(scales, 128, axis=1).astype(np.float64)
    assert np.all(np.abs(y - x) <= np.abs(x) * (2.0 ** -4 + 2.0 ** -8) + sc * 2.0 ** -9 + 1e-30)


def test_sparse_mla_reads_the_quantised_rows_as_their_dequantised_values():
    # attention over fp8 rows (read through their scales) equals attention over the
    # bf16 rows the dequantiser writes, up to that final bf16 rounding
    rng = np.random.default_rng(16)
    n, H, k = 40, 4, 32
    lat = _rows(rng, n, 512)
    rope = _bf16_of(rng.standard_normal((n, 64)).astype(np.float32))
    rows = oracle.quantize_mla_rows(lat, rope)
    back = oracle.dequantize_mla_rows(rows, 512, 64)
    q_nope = _bf16_of(rng.standard_normal((1, H, 512)).astype(np.float32) * 0.05)
    q_rope = _bf16_of(rng.standard_normal((1, H, 64)).astype(np.float32) * 0.05)
    idx = rng.permutation(n)[:k].astype(np.int32)[None, :]
    o8, l8 = oracle.sparse_mla(W.DT_BF16, W.DT_E4M3, q_nope, q_rope, rows, idx, 0.07)
    ob, lb = oracle.sparse_mla(W.DT_BF16, W.DT_BF16, q_nope, q_rope, back, idx, 0.07)
    assert np.allclose(o8, ob, rtol=0, atol=2e-2 * (1 + np.abs(ob)).max())
    assert np.allclose(l8, lb, rtol=0, atol=1e-2)


# ------------------------------------------------------------------ RAGGED extend

def test_ragged_topk_is_the_paged_topk_through_an_offset_identity_table():
    # RAGGED indices = positions + the request's offset; the paged transform through a
    # page table that maps position s to offset + s gives the same row
    rng = np.random.default_rng(21)
    B, Wd, k = 3, 500, 64
    lens = np.array([400, 30, 500], np.int32)
    offsets = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32)
    lg = rng.standard_normal((B, Wd)).astype(np.float32)
    lg[0, ::5] = 1.0  # ties
    r2q = np.arange(B, dtype=np.int32)
    rag = oracle.topk_ragged(lg, lens, r2q, offsets, k)
    table = offsets[:, None] + np.arange(Wd, dtype=np.int32)[None, :]
    assert np.array_equal(rag, oracle.topk_transform(lg, lens, r2q, table, k))
    # the pages' formula: where(idx != -1, idx + offset, idx) on the position top-k
    pos = oracle.topk_transform(lg, lens, r2q, np.tile(np.arange(Wd, dtype=np.int32), (B, 1)), k)
    assert np.array_equal(rag, np.where(pos != -1, pos + offsets[:, None], pos))
    assert np.all(rag[1, 30:] == -1) and np.array_equal(rag[1, :30], offsets[1] + np.arange(30))


def test_flatten_page_table_is_the_concatenation_of_live_prefixes():
    rng = np.random.default_rng(22)
    pt = rng.integers(0, 10 ** 6, size=(4, 50)).astype(np.int32)
    kv = np.array([50, 0, 17, 33], np.int32)
    flat = oracle.flatten_page_table(pt, kv)
    assert np.array_equal(flat, np.concatenate([pt[b, :kv[b]] for b in range(4)]))
