"""Pins of the oracle's chunk-local dense attention (CPU only).

(1) One virtual batch holding the whole sequence is plain causal attention:
    compared with PyTorch's scaled_dot_product_attention in float64 (GQA heads
    repeated, the causal mask aligned to the end of the keys).
(2) The whole local-attention path — make_local_attention_virtual_batches, then
    attention per virtual batch through its local block table — equals dense
    attention in which the query at absolute position p sees the keys of its own
    chunk up to p, written here directly over each request's contiguous keys."""
import numpy as np
import pytest
import torch

import oracle


def _bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def _paged(rng, kv_lens, ps, Hkv, D, slack=3):
    """Per-request keys/values in a shuffled page pool: caches [pages, ps, Hkv, D] and
    block tables [B, max_pages] (request-relative pages)."""
    pages_per = [(int(L) + ps - 1) // ps for L in kv_lens]
    total = sum(pages_per) + slack
    perm = rng.permutation(total)
    kc = _bf16(rng, (total, ps, Hkv, D))
    vc = _bf16(rng, (total, ps, Hkv, D))
    bt = np.full((len(kv_lens), max(pages_per) + 2), -1, np.int32)
    k = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[k:k + n]
        k += n
    return kc, vc, bt


def test_single_chunk_is_causal_sdpa():
    rng = np.random.default_rng(41)
    Hq, Hkv, D, ps = 8, 2, 64, 16
    kv_lens = np.array([50, 17, 96], np.int32)
    q_lens = np.array([5, 17, 1], np.int32)
    kc, vc, bt = _paged(rng, kv_lens, ps, Hkv, D)
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _bf16(rng, (int(cq[-1]), Hq, D))
    scale = D ** -0.5
    out, lse = oracle.local_attention(q, kc, vc, bt, cq, kv_lens, scale)
    for b in range(3):
        L, n = int(kv_lens[b]), int(q_lens[b])
        slots = bt[b, np.arange(L) // ps] * ps + np.arange(L) % ps
        K = _f64(kc.reshape(-1, Hkv, D)[slots])          # [L, Hkv, D]
        V = _f64(vc.reshape(-1, Hkv, D)[slots])
        Q = _f64(q[cq[b]:cq[b + 1]])                      # [n, Hq, D]
        rep = Hq // Hkv
        Kt = torch.from_numpy(K).repeat_interleave(rep, dim=1).permute(1, 0, 2)  # [Hq, L, D]
        Vt = torch.from_numpy(V).repeat_interleave(rep, dim=1).permute(1, 0, 2)
        Qt = torch.from_numpy(Q).permute(1, 0, 2)                                # [Hq, n, D]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]    # [n, L]
        ref = torch.nn.functional.scaled_dot_product_attention(Qt, Kt, Vt, attn_mask=mask, scale=scale)
        assert np.allclose(out[cq[b]:cq[b + 1]], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
        logits = (Qt @ Kt.transpose(1, 2)) * scale
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1).T
        assert np.allclose(lse[cq[b]:cq[b + 1]], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_local_virtual_batches_path_is_chunked_causal_attention(seed):
    rng = np.random.default_rng(50 + seed)
    Hq, Hkv, D = 4, 2, 32
    ps = int(rng.choice([2, 4, 8]))
    chunk = ps * int(rng.integers(1, 5))
    B = int(rng.integers(1, 4))
    kv_lens = rng.integers(1, 60, size=B).astype(np.int32)
    q_lens = np.array([int(rng.integers(1, L + 1)) for L in kv_lens], np.int32)
    kc, vc, bt = _paged(rng, kv_lens, ps, Hkv, D, slack=1)
    # block tables wide enough for the last chunk of every request
    bt = np.concatenate([bt, np.full((B, chunk // ps + 1), 0, np.int32)], axis=1)
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _bf16(rng, (int(cq[-1]), Hq, D))
    sq, cu_local, sk, starts, bt_local = oracle.local_virtual_batches(chunk, ps, cq, kv_lens, bt)
    out, lse = oracle.local_attention(q, kc, vc, bt_local, cu_local, sk, 0.3)
    # direct statement: query at absolute position p of request b sees keys floor(p/c)*c .. p
    exp_out = np.zeros_like(out)
    exp_lse = np.zeros_like(lse)
    for b in range(B):
        L, n = int(kv_lens[b]), int(q_lens[b])
        slots = bt[b, np.arange(L) // ps] * ps + np.arange(L) % ps
        K = _f64(kc.reshape(-1, Hkv, D)[slots])
        V = _f64(vc.reshape(-1, Hkv, D)[slots])
        for i in range(n):
            t = cq[b] + i
            pos = L - n + i
            lo = (pos // chunk) * chunk
            for h in range(Hq):
                qh = _f64(q[t, h])
                s = 0.3 * (K[lo:pos + 1, h // (Hq // Hkv)] @ qh)
                m = s.max()
                w = np.exp(s - m)
                exp_lse[t, h] = m + np.log(w.sum())
                exp_out[t, h] = (w / w.sum()) @ V[lo:pos + 1, h // (Hq // Hkv)]
    assert np.allclose(out, exp_out, rtol=1e-10, atol=1e-12)
    assert np.allclose(lse, exp_lse, rtol=1e-12, atol=1e-12)
