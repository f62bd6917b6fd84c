"""One step of the sparse-attention path on one GPU: metadata -> indexer
logits -> top-k + slot transform -> sparse MLA, through the C ABI.

`SparseAttentionStep` owns the device buffers of one step (inputs, metadata,
logits, indices, outputs, scratch) and enqueues the four library calls.
The inputs come from any object with the attributes documented in
`from_host` (numpy arrays); nothing here computes any part of the path.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import (DT_BF16, MODE_EXTEND, alloc_metadata, alloc_score_hist, alloc_topk_workspace,
               nsa_indexer_logits, nsa_metadata, nsa_sparse_mla, nsa_sparse_mla_workspace_bytes, nsa_status_read,
               nsa_topk_transform, nsa_topk_workspace_bytes)


def _dev(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


class SparseAttentionStep:
    """Device state of one step.

    Host inputs (numpy), read by `from_host`:
      mode, B, R, W, n_draft, topk, page_size, seq_lens [B], extend_lens [B] | None,
      req_to_token [pool, W'], req_pool_indices [B], idx_dtype, q_idx [R,Hi,Di] (uint8 e4m3 or
      float32), weights [R,Hi], k_cache [pages, ps, Di], k_scale [pages, ps], q_dtype, kv_dtype,
      q_nope [R,H,d_latent], q_rope [R,H,d_rope] (bf16 bits as uint16, or float32),
      kv [slots, row] (bf16 bits / e4m3 row bytes / float32), sm_scale.
    """

    def __init__(self, host, device="cuda", fuse_topk: Optional[bool] = None, page_table_1: bool = False):
        """fuse_topk: the indexer counts each row's leading score digits for the top-k
        (the indexer-to-top-k fusion); False: the top-k counts them itself.  Default:
        fused when the rows are long enough for the top-k to select them in chunks over
        several CTAs (it then needs a workspace), where the counts save it a pass over
        the scores; unfused when every row fits one CTA, which counts its cached row
        more cheaply than the indexer's epilogue can.
        page_table_1: the metadata also copies the requests' req_to_token rows into
        page_table_1 and the top-k reads the slots from there; False (default): no copy,
        the top-k reads them from req_to_token through the metadata's req_rows."""
        self.h = host
        self.device = torch.device(device)
        d = self.device
        self.mode, self.B, self.R, self.W = host.mode, host.B, host.R, host.W
        self.topk, self.ps, self.n_draft = host.topk, host.page_size, host.n_draft
        self.idx_dtype, self.q_dtype, self.kv_dtype = host.idx_dtype, host.q_dtype, host.kv_dtype
        self.sm_scale = float(host.sm_scale)
        # rows sharing a request are scored together (decode 1, verify n_draft, extend 4)
        self.rows_per_group = {0: 1, 1: 4, 2: max(1, min(4, self.n_draft))}[self.mode]
        self.seq_lens = _dev(host.seq_lens.astype(np.int32), d)
        self.extend_lens = None if host.extend_lens is None else _dev(host.extend_lens.astype(np.int32), d)
        self.req_to_token = _dev(host.req_to_token, d)
        self.req_pool_indices = _dev(host.req_pool_indices, d)
        self.q_idx = _dev(host.q_idx, d)
        self.weights = _dev(host.weights, d)
        self.k_cache = _dev(host.k_cache, d)
        self.k_scale = _dev(host.k_scale, d)
        bf = torch.bfloat16
        self.q_nope = _dev(host.q_nope.view(np.int16), d, bf) if self.q_dtype == DT_BF16 else _dev(host.q_nope, d)
        self.q_rope = _dev(host.q_rope.view(np.int16), d, bf) if self.q_dtype == DT_BF16 else _dev(host.q_rope, d)
        self.kv = _dev(host.kv.view(np.int16), d, bf) if self.kv_dtype == DT_BF16 else _dev(host.kv, d)
        self.num_slots = int(host.kv.shape[0])
        self.H, self.d_latent, self.d_rope = host.q_nope.shape[1], host.q_nope.shape[2], host.q_rope.shape[2]
        self.md = alloc_metadata(self.mode, self.B, self.R, self.W, self.ps, d, with_ks_ke=self.mode == MODE_EXTEND,
                                 with_page_table_1=page_table_1, with_req_rows=True)
        self.logits_ld = max(4, (self.W + 3) // 4 * 4)
        self.logits = torch.empty((self.R, self.logits_ld), dtype=torch.float32, device=d)
        self.indices = torch.empty((self.R, self.topk), dtype=torch.int32, device=d)
        if fuse_topk is None:
            fuse_topk = nsa_topk_workspace_bytes(self.R, self.W, False) > 0
        self.score_hist = alloc_score_hist(self.R, d) if fuse_topk else None
        self.topk_ws = alloc_topk_workspace(self.R, self.W, fuse_topk, d)
        odt = torch.bfloat16 if self.q_dtype == DT_BF16 else torch.float32
        self.out = torch.empty((self.R, self.H, self.d_latent), dtype=odt, device=d)
        self.lse = torch.empty((self.R, self.H), dtype=torch.float32, device=d)
        ws = nsa_sparse_mla_workspace_bytes(self.q_dtype, self.kv_dtype, self.R, self.H, self.d_latent,
                                            self.d_rope, self.topk)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=d) if ws > 0 else None
        self.status = torch.zeros(1, dtype=torch.int32, device=d)

    # ---------------------------------------------------------- stages
    def metadata(self, stream=None, seq_lens: Optional[torch.Tensor] = None,
                 req_pool_indices: Optional[torch.Tensor] = None, extend_lens: Optional[torch.Tensor] = None):
        """seq_lens / req_pool_indices / extend_lens default to the step's device copies;
        pinned host tensors (mapped into the device's address space) are read directly."""
        nsa_metadata(self.mode, self.B, self.R, self.W, self.n_draft, self.topk, self.ps,
                     self.seq_lens if seq_lens is None else seq_lens,
                     self.extend_lens if extend_lens is None else extend_lens, self.req_to_token,
                     self.req_pool_indices if req_pool_indices is None else req_pool_indices, self.md,
                     self.status, stream)

    def indexer(self, stream=None):
        nsa_indexer_logits(self.idx_dtype, self.q_idx, self.weights, self.k_cache, self.k_scale,
                           self.md["real_page_table"], self.md["row_to_req"], self.md["seqlens_expanded"],
                           self.W, self.logits, self.status, stream, rows_per_group=self.rows_per_group,
                           score_hist=self.score_hist)

    def topk_transform(self, stream=None, logits: Optional[torch.Tensor] = None):
        """With other `logits` than the indexer's the histogram does not describe them:
        the top-k then counts the digits itself (and still clears the buffer)."""
        copied = "page_table_1" in self.md
        nsa_topk_transform(self.logits if logits is None else logits, self.md["seqlens_expanded"],
                           self.md["row_to_req"], self.md["page_table_1"] if copied else self.req_to_token,
                           self.topk, self.W, self.indices, self.status, stream, score_hist=self.score_hist,
                           workspace=self.topk_ws, pt_rows=None if copied else self.md["req_rows"])

    def attention(self, stream=None, indices: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None):
        """out / lse default to the step's device buffers; pinned host tensors (mapped
        into the device's address space) receive the result directly."""
        nsa_sparse_mla(self.q_dtype, self.kv_dtype, self.q_nope, self.q_rope, self.kv,
                       self.indices if indices is None else indices, self.sm_scale,
                       self.out if out is None else out, self.lse if lse is None else lse,
                       self.workspace, self.status, stream, num_slots=self.num_slots)

    def run(self, stream=None):
        """Enqueue the whole step (4 library calls)."""
        self.metadata(stream)
        self.indexer(stream)
        self.topk_transform(stream)
        self.attention(stream)

    def status_code(self, stream=None) -> int:
        return nsa_status_read(self.status, stream)
