"""KV-cache write side on the GPU vs the oracle, through the C ABI: every
written byte (e4m3 codes, fp32 scales, bf16 values) bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_sparse_mla_indexer_gb300 as nsa
    nsa.load()


def _bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rows(rng, n):
    lat = _bf16(rng, (n, 512))
    lat[0, :128] = 0                                   # all-zero block
    lat[1, 200] = np.uint16(0x4280)                    # 64.0: an outlier
    lat[2] = _bf16(rng, (512,), 1e-6)                  # tiny values
    lat[3, 384:] = np.uint16(0x8000)                   # a block of -0.0
    rope = _bf16(rng, (n, 64))
    return lat, rope


def _t(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


@pytest.mark.parametrize("n,pool", [(1, 8), (300, 1000), (4097, 5000)])
def test_set_mla_kv_fp8_rows_bit_exact(n, pool):
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(n)
    lat, rope = _rows(rng, max(n, 4))
    lat, rope = lat[:n], rope[:n]
    loc = rng.choice(pool, size=n, replace=False).astype(np.int32)
    kv = torch.full((pool, 656), 0xA5, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nsa.nsa_set_mla_kv(nsa.DT_E4M3, _t(lat, torch.int16), _t(rope, torch.int16), _t(loc), kv, status)
    got = kv.cpu().numpy()
    assert status.item() == 0
    assert np.array_equal(got[loc], oracle.quantize_mla_rows(lat, rope))
    untouched = np.setdiff1d(np.arange(pool), loc)
    assert np.all(got[untouched] == 0xA5)


def test_set_mla_kv_bf16_rows_copied():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(2)
    lat, rope = _rows(rng, 64)
    loc = rng.permutation(100)[:64].astype(np.int32)
    kv = torch.zeros((100, 576), dtype=torch.int16, device="cuda")
    nsa.nsa_set_mla_kv(nsa.DT_BF16, _t(lat, torch.int16), _t(rope, torch.int16), _t(loc), kv)
    got = kv.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[loc], np.concatenate([lat, rope], axis=1))


def test_quantize_whole_cache_bit_exact():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(3)
    lat, rope = _rows(rng, 3000)
    cache = np.concatenate([lat, rope], axis=1)
    out = torch.empty((3000, 656), dtype=torch.uint8, device="cuda")
    nsa.nsa_quantize_kv_cache(_t(cache, torch.int16), out)
    assert np.array_equal(out.cpu().numpy(), oracle.quantize_mla_rows(lat, rope))


def test_quantize_full_size_cache_sampled_rows():
    # the bf16 KV cache of the 32-request decode workload (every slot), rows sampled
    import deepseek_sparse_mla_indexer_gb300 as nsa
    wl = W.config("v32_decode_bf16")
    n = wl.kv.shape[0]
    out = torch.empty((n, 656), dtype=torch.uint8, device="cuda")
    nsa.nsa_quantize_kv_cache(_t(wl.kv.view(np.int16)), out)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 500)]))
    kvb = wl.kv.view(np.uint16)
    exp = oracle.quantize_mla_rows(kvb[rows, :512], kvb[rows, 512:])
    assert np.array_equal(out.cpu().numpy()[rows], exp)


def test_dequantize_paged_bit_exact_with_padding_and_bounds():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(5)
    lat, rope = _rows(rng, 500)
    fp8 = oracle.quantize_mla_rows(lat, rope)
    slots = rng.integers(0, 500, 777).astype(np.int32)
    slots[::50] = -1               # padding: zero rows, no error
    out = torch.full((777, 576), 7, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nsa.nsa_dequantize_kv_paged(_t(fp8), _t(slots), out, status=status)
    got = out.cpu().numpy().view(np.uint16)
    valid = slots >= 0
    assert status.item() == 0
    assert np.array_equal(got[valid], oracle.dequantize_mla_rows(fp8[slots[valid]], 512, 64))
    assert not got[~valid].any()
    slots[3] = 500                 # one past the end
    status.zero_()
    nsa.nsa_dequantize_kv_paged(_t(fp8), _t(slots), out, status=status)
    assert status.item() == nsa.ERR_BOUNDS
    assert not out[3].any().item()


@pytest.mark.parametrize("n", [1, 333, 2048])
def test_set_index_k_bit_exact(n):
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(100 + n)
    k = _bf16(rng, (n, 128))
    k[0, :] = 0
    pool = 4096
    loc = rng.choice(pool, size=n, replace=False).astype(np.int32)
    kc = torch.zeros((pool, 128), dtype=torch.uint8, device="cuda")
    ks = torch.full((pool,), -1.0, dtype=torch.float32, device="cuda")
    nsa.nsa_set_index_k(_t(k, torch.int16), _t(loc), kc, ks)
    codes, scales = oracle.quantize_index_rows(k)
    assert np.array_equal(kc.cpu().numpy()[loc], codes)
    assert np.array_equal(ks.cpu().numpy()[loc], scales)
    untouched = np.setdiff1d(np.arange(pool), loc)
    assert np.all(ks.cpu().numpy()[untouched] == -1.0)


def test_out_of_range_slot_sets_bounds_and_is_skipped():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(6)
    lat, rope = _rows(rng, 4)
    loc = np.array([0, 9, 2, -3], np.int32)  # 9 and -3 lie outside a pool of 4
    kv = torch.zeros((4, 656), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nsa.nsa_set_mla_kv(nsa.DT_E4M3, _t(lat, torch.int16), _t(rope, torch.int16), _t(loc), kv, status)
    assert status.item() == nsa.ERR_BOUNDS
    got = kv.cpu().numpy()
    exp = oracle.quantize_mla_rows(lat, rope)
    assert np.array_equal(got[0], exp[0]) and np.array_equal(got[2], exp[2])
    assert not got[1].any() and not got[3].any()


def test_host_rejects_bad_arguments():
    import deepseek_sparse_mla_indexer_gb300 as nsa
    k = torch.zeros((4, 64), dtype=torch.int16, device="cuda")  # Di 64 is not supported
    with pytest.raises(nsa.NsaError):
        nsa.nsa_set_index_k(k, torch.zeros(4, dtype=torch.int32, device="cuda"),
                            torch.zeros((8, 64), dtype=torch.uint8, device="cuda"),
                            torch.zeros(8, dtype=torch.float32, device="cuda"))
    lat = torch.zeros((4, 256), dtype=torch.int16, device="cuda")  # d_latent 256 is not supported
    with pytest.raises(nsa.NsaError):
        nsa.nsa_set_mla_kv(nsa.DT_E4M3, lat, torch.zeros((4, 64), dtype=torch.int16, device="cuda"),
                           torch.zeros(4, dtype=torch.int32, device="cuda"),
                           torch.zeros((8, 656), dtype=torch.uint8, device="cuda"))


def test_copy_buffers_between_pinned_host_and_device():
    # several copies in one launch, host inputs in and device results out, bit-exact
    import deepseek_sparse_mla_indexer_gb300 as nsa
    rng = np.random.default_rng(9)
    sizes = [16, 4096, 12345, 1 << 20, 0, 48]
    hsrc = [torch.from_numpy(rng.integers(0, 255, n, dtype=np.uint8)).pin_memory() for n in sizes]
    dev = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in sizes]
    nsa.nsa_copy_buffers(list(zip(dev, hsrc)))
    back = [torch.empty(n, dtype=torch.uint8).pin_memory() for n in sizes]
    nsa.nsa_copy_buffers(list(zip(back, dev)))
    torch.cuda.synchronize()
    for a, b in zip(hsrc, back):
        assert torch.equal(a, b)
    # 16-byte aligned sizes take the vector path
    a16 = torch.from_numpy(rng.integers(0, 255, 1 << 16, dtype=np.uint8)).pin_memory()
    d16 = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    nsa.nsa_copy_buffers([(d16, a16)])
    torch.cuda.synchronize()
    assert torch.equal(d16.cpu(), a16)
    # pageable host memory is refused, not touched
    with pytest.raises(nsa.NsaError):
        nsa.nsa_copy_buffers([(d16, torch.zeros(1 << 16, dtype=torch.uint8))])
