"""Device-resident state of one decode workload, built from the seeded inputs.

Uploads the seeded queries and weights, allocates the paged cache pool, and
writes every sequence into it with ``mla_cache_fill`` (NaN-poisoned tail
slots).  ``step()`` runs one decode step through the four C-ABI calls.
"""
from __future__ import annotations

import numpy as np
import torch

import mla_inputs as mi

from . import binding as C


def storage_to_torch(a: np.ndarray, dtype: str, device) -> torch.Tensor:
    """numpy storage array (bf16 bits as uint16, or float32) -> torch tensor on device."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    elif dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    else:
        raise ValueError(dtype)
    return t.to(device)


class DeviceWorkload:
    """Everything one decode step reads and writes, resident on one GPU."""

    def __init__(self, w: mi.Workload, device="cuda", num_parts: int | None = None,
                 rows_per_upload: int = 1 << 20, out_dtype=torch.float32,
                 fill_lens: np.ndarray | None = None, q_len: int = 1):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        lens = mi.lengths(w)
        table, nblk = mi.block_table(w, lens)
        self.lens_np = lens
        # rows written at set-up (the rest are appended by append_tail)
        self.fill_np = lens.copy() if fill_lens is None else np.minimum(
            np.asarray(fill_lens, dtype=np.int64), lens)
        self.table_np = table
        self.num_blocks = nblk
        self.max_len = int(lens.max())
        tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16

        # q_len new tokens per sequence: queries [B, q_len, h, .] at positions
        # L_b - q_len + j (q_len = 1 keeps the one-token shapes [B, h, .])
        self.q_len = int(q_len)
        if self.q_len == 1:
            qn, qr = mi.queries(w)
        else:
            qn, qr = mi.queries_multi(w, self.q_len)
        wuk, wuv = mi.weights(w)
        self.q_nope = storage_to_torch(qn, w.dtype, dev)
        self.q_rope = storage_to_torch(qr, w.dtype, dev)
        self.w_uk = storage_to_torch(wuk, w.dtype, dev)
        self.w_uv = storage_to_torch(wuv, w.dtype, dev)
        self.q_pos = torch.from_numpy(
            mi.query_positions(w, lens) if self.q_len == 1 else
            mi.query_positions_multi(w, self.q_len, lens)).to(dev)
        self.seq_lens = torch.from_numpy(lens.astype(np.int32)).to(dev)
        self.block_table = torch.from_numpy(table).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

        # cache pool, tails poisoned with NaN
        bs, d_c, d_r = w.block_size, w.d_c, w.d_r
        if w.latent_dtype == "fp8e4m3":
            self.latent = torch.full((nblk, bs, d_c), 0x7F, dtype=torch.uint8, device=dev)
            self.rope = torch.full((nblk, bs, d_r), float("nan"), dtype=torch.bfloat16, device=dev)
            self.scale = torch.full((nblk,), float("nan"), dtype=torch.float32, device=dev)
            self.kv = C.KVCache.split(self.latent, self.rope, self.scale)
            self.pool = None
        else:
            self.pool = torch.full((nblk, bs, d_c + d_r), float("nan"), dtype=tdt, device=dev)
            self.kv = C.KVCache.packed(self.pool, d_c, d_r)
        self._fill(rows_per_upload)

        if num_parts is None:
            num_parts = C.default_num_parts(dev)
        self.num_parts = int(num_parts)
        B, h = w.B, w.h
        nslot = C.mla_decode_num_partials(B, self.num_parts)
        lead = (B,) if self.q_len == 1 else (B, self.q_len)
        rows = self.q_len * h
        self.q_cat = torch.empty(lead + (h, d_c + d_r), dtype=tdt, device=dev)
        self.o_part = torch.empty((nslot, rows, d_c), dtype=torch.float32, device=dev)
        self.lse_part = torch.empty((nslot, rows), dtype=torch.float32, device=dev)
        self.o_lat = torch.empty(lead + (h, d_c), dtype=tdt, device=dev)
        self.lse = torch.empty(lead + (h,), dtype=torch.float32, device=dev)
        self.out = torch.empty(lead + (h, w.d_v), dtype=out_dtype, device=dev)

    # -- cache -------------------------------------------------------------
    def _fill(self, rows_per_upload: int) -> None:
        w = self.w
        src_dt = mi.latent_source_dtype(w)
        b = 0
        fl = self.fill_np
        while b < w.B:
            e, rows = b, 0
            while e < w.B and (e == b or rows + fl[e] <= rows_per_upload):
                rows += int(fl[e])
                e += 1
            if rows == 0:
                b = e
                continue
            cs, krs = [], []
            for bb in range(b, e):
                c, kr = mi.sequence(w, bb, int(self.lens_np[bb]))
                cs.append(c[: fl[bb]])
                krs.append(kr[: fl[bb]])
            c_t = storage_to_torch(np.concatenate(cs), src_dt, self.device)
            kr_t = storage_to_torch(np.concatenate(krs), w.dtype, self.device)
            cu = np.zeros(e - b + 1, dtype=np.int32)
            cu[1:] = np.cumsum(fl[b:e])
            cu_t = torch.from_numpy(cu).to(self.device)
            tab = self.block_table[b:e].contiguous()
            C.mla_cache_fill(c_t, kr_t, cu_t, int(max(1, fl[b:e].max())), tab, self.kv,
                             rope_theta=w.theta, dev_status=self.status)
            b = e
        torch.cuda.synchronize(self.device)

    def append_tail(self) -> int:
        """Append the rows past the set-up fill one token per call: call s
        appends row fill_b + s of every sequence that still has one, through
        mla_cache_append.  Returns the number of calls."""
        w = self.w
        src_dt = mi.latent_source_dtype(w)
        todo = self.lens_np - self.fill_np
        seqs = {b: mi.sequence(w, b, int(self.lens_np[b])) for b in range(w.B) if todo[b] > 0}
        calls = 0
        for step in range(int(todo.max()) if len(todo) else 0):
            bs = [b for b in range(w.B) if todo[b] > step]
            t = [int(self.fill_np[b]) + step for b in bs]
            c = np.stack([seqs[b][0][tt] for b, tt in zip(bs, t)])
            kr = np.stack([seqs[b][1][tt] for b, tt in zip(bs, t)])
            idx = torch.tensor(bs, dtype=torch.long, device=self.device)
            C.mla_cache_append(storage_to_torch(c, src_dt, self.device),
                               storage_to_torch(kr, w.dtype, self.device),
                               torch.tensor(t, dtype=torch.int32, device=self.device),
                               self.block_table.index_select(0, idx).contiguous(), self.kv,
                               rope_theta=w.theta, dev_status=self.status)
            calls += 1
        torch.cuda.synchronize(self.device)
        return calls

    # -- the hidden-state boundary -----------------------------------------
    def enable_hidden(self, d_model: int, d_cq: int) -> None:
        """Upload the hidden state x and the linear layers around the step
        (query compression W_DQ, W_UQ, W_QR; output projection W_O) and the
        buffers of query_from_hidden / hidden_out."""
        w = self.w
        assert self.q_len == 1 and w.dtype == "bf16"
        hid = mi.hidden_inputs(w, d_model, d_cq)
        for k, v in hid.items():
            setattr(self, k, storage_to_torch(v, w.dtype, self.device))
        dev, B, h = self.device, w.B, w.h
        self.d_model, self.d_cq = d_model, d_cq
        self.c_q = torch.empty((B, d_cq), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((B, d_model), dtype=torch.float32, device=dev)
        self.out_bf16 = torch.empty((B, h, w.d_v), dtype=torch.bfloat16, device=dev)
        self.w_fold = None
        ws = max(C.mla_linear_workspace_bytes(B, d_model, d_cq),
                 C.mla_linear_workspace_bytes(B, d_cq, h * w.d_nope),
                 C.mla_linear_workspace_bytes(B, d_cq, h * w.d_r),
                 C.mla_linear_workspace_bytes(B, h * w.d_v, d_model),
                 C.mla_linear_workspace_bytes(B, h * w.d_c, d_model))
        self.lin_ws = torch.empty(max(1, ws // 4), dtype=torch.float32, device=dev)

    def query_from_hidden(self, stream=None):
        """q_nope, q_rope <- the compressed query of x (three linear layers)."""
        w = self.w
        B = w.B
        C.mla_linear(self.x, self.w_dq, self.c_q, self.lin_ws, stream)
        C.mla_linear(self.c_q, self.w_uq, self.q_nope.view(B, -1), self.lin_ws, stream)
        C.mla_linear(self.c_q, self.w_qr, self.q_rope.view(B, -1), self.lin_ws, stream)

    def hidden_out(self, folded: bool = False, stream=None):
        """y <- the step's output projected to the hidden size: W_UV then W_O
        (folded=False), or the merged W_O W_UV applied to o_lat (folded=True)."""
        w = self.w
        B = w.B
        if folded:
            if self.w_fold is None:
                self.w_fold = torch.empty((self.d_model, w.h * w.d_c), dtype=torch.bfloat16,
                                          device=self.device)
                C.mla_fold_uv_into_o(self.w_uv, self.w_o, self.w_fold, stream)
            C.mla_linear(self.o_lat.view(B, -1), self.w_fold, self.y, self.lin_ws, stream)
        else:
            C.mla_out_proj(self.o_lat, self.w_uv, self.out_bf16, stream=stream)
            C.mla_linear(self.out_bf16.view(B, -1), self.w_o, self.y, self.lin_ws, stream)

    def hidden_step(self, folded: bool = False, stream=None):
        """The whole step from the hidden state x to the output hidden state y."""
        self.query_from_hidden(stream)
        self.absorb(stream)
        self.attend(stream=stream)
        self.combine(stream)
        self.hidden_out(folded, stream)
        return self.y

    # -- the decode step ---------------------------------------------------
    def _rows(self, t: torch.Tensor) -> torch.Tensor:
        """[B, q_len, h, .] -> [B * q_len, h, .] (the per-token calls' view)."""
        return t if self.q_len == 1 else t.reshape((-1,) + tuple(t.shape[2:]))

    def absorb(self, stream=None):
        C.mla_absorb_q(self._rows(self.q_nope), self._rows(self.q_rope), self.q_pos.reshape(-1),
                       self.w_uk, self._rows(self.q_cat), rope_theta=self.w.theta, stream=stream)

    def attend(self, flags=C.MLA_DECODE_AUTO, stream=None):
        if self.q_len == 1:
            C.mla_decode_fwd(self.q_cat, self.kv, self.block_table, self.seq_lens,
                             self.num_parts, self.o_part, self.lse_part, dev_status=self.status,
                             flags=flags, stream=stream)
        else:
            C.mla_decode_fwd_multi(self.q_cat, self.kv, self.block_table, self.seq_lens,
                                   self.num_parts, self.o_part, self.lse_part,
                                   dev_status=self.status, flags=flags, stream=stream)

    def combine(self, stream=None):
        B = self.w.B
        C.mla_combine(self.o_part, self.lse_part, self.seq_lens, self.w.block_size,
                      self.block_table.shape[1], self.num_parts,
                      self.o_lat.view(B, -1, self.w.d_c), self.lse.view(B, -1), stream=stream)

    def project(self, stream=None):
        C.mla_out_proj(self._rows(self.o_lat), self.w_uv, self._rows(self.out), stream=stream)

    # The merge and W_UV as one kernel (mla_combine_out_proj) is available for
    # one-token steps over bf16 weights; the step uses the pair of kernels,
    # which measured faster at the V3 shapes (28.7 against 36.7 us).
    fuse_tail = False

    @property
    def fused_tail(self) -> bool:
        return self.fuse_tail and self.q_len == 1 and self.w_uv.dtype == torch.bfloat16

    def combine_project(self, stream=None):
        """mla_combine and mla_out_proj in one call; o_lat and lse are written too."""
        C.mla_combine_out_proj(self.o_part, self.lse_part, self.seq_lens, self.w.block_size,
                               self.block_table.shape[1], self.num_parts, self.w_uv, self.out,
                               o_lat=self.o_lat, lse=self.lse, dev_status=self.status,
                               stream=stream)

    def tail(self, stream=None):
        """The step after the decode: merged kernel where it applies, else the pair."""
        if self.fused_tail:
            self.combine_project(stream)
        else:
            self.combine(stream)
            self.project(stream)

    def launches_per_step(self) -> int:
        return 3 if self.fused_tail else 4

    def step(self, flags=C.MLA_DECODE_AUTO, stream=None):
        self.absorb(stream)
        self.attend(flags, stream)
        self.tail(stream)
        return self.out

    # -- bookkeeping -------------------------------------------------------
    def cache_bytes(self) -> float:
        """Algorithmic bytes of the cache one step reads: sum_b L_b * bytes/token."""
        w = self.w
        per_tok = C.mla_cache_bytes_per_token(
            {"f32": 0, "bf16": 1, "fp8e4m3": 2}[w.latent_dtype],
            0 if w.dtype == "f32" else 1, w.d_c, w.d_r, w.block_size)
        return float(self.lens_np.sum()) * per_tok

    def step_bytes(self) -> float:
        """Algorithmic bytes of one full step (cache, queries, weights, outputs)."""
        w = self.w
        el = 4 if w.dtype == "f32" else 2
        B, h = w.B, w.h
        q_in = B * self.q_len * h * (w.d_nope + w.d_r) * el
        wts = 2 * h * w.d_v * w.d_c * el
        table = self.table_np.size * 4 + B * 4
        out = B * self.q_len * h * w.d_v * self.out.element_size()
        return self.cache_bytes() + q_in + wts + table + out

    def decode_bytes(self) -> float:
        """Algorithmic bytes of one mla_decode_fwd launch: every cached token
        once, the absorbed queries, the block table and the lengths."""
        w = self.w
        el = 4 if w.dtype == "f32" else 2
        return (self.cache_bytes() + w.B * self.q_len * w.h * (w.d_c + w.d_r) * el
                + self.table_np.size * 4 + w.B * 4)

    def decode_flops(self) -> float:
        """2 * h * (d_c + d_r) score flops plus 2 * h * d_c P.C flops per cached token
        and query token (the masked corner of the causal triangle is not removed)."""
        w = self.w
        return float(self.lens_np.sum()) * self.q_len * w.h * 2 * (w.d_c + w.d_r + w.d_c)

    def step_flops(self) -> float:
        """2 * h * (d_c + d_r + d_c) per cached token, plus the two per-head GEMMs."""
        w = self.w
        attn = float(self.lens_np.sum()) * self.q_len * w.h * 2 * (w.d_c + w.d_r + w.d_c)
        gemms = 2.0 * w.B * self.q_len * w.h * w.d_c * (w.d_nope + w.d_v)
        return attn + gemms

    def check_status(self) -> int:
        return int(self.status.item())


class DevicePrefill:
    """A prompt prefill of a workload's sequences in the MHA form, resident on
    one GPU: the latent rows and rotated RoPE keys (written to the paged cache
    and gathered back bit for bit), the per-head keys and values
    k_nope = c W_UK^T and v = c W_UV^T (mla_linear), the queries
    (mla_prefill_query) and the causal attention (mla_prefill_fwd)."""

    def __init__(self, w: mi.Workload, device="cuda", out_dtype=torch.float32):
        self.w = w
        self.dw = DeviceWorkload(w, device=device)
        dev = self.dw.device
        lens = self.dw.lens_np
        self.device = dev
        self.lens_np = lens
        self.T = int(lens.sum())
        self.max_len = int(lens.max())
        cu = np.zeros(w.B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        self.cu = torch.from_numpy(cu).to(dev)
        h = w.h
        self.c = torch.empty((self.T, w.d_c), dtype=torch.bfloat16, device=dev)
        self.k_rope = torch.empty((self.T, w.d_r), dtype=torch.bfloat16, device=dev)
        C.mla_paged_gather(self.dw.kv, self.dw.block_table, self.cu, self.max_len, self.c,
                           self.k_rope, dev_status=self.dw.status)
        qn, qr = mi.prefill_queries(w, lens)
        self.q_nope = storage_to_torch(qn, w.dtype, dev)
        self.q_rope = storage_to_torch(qr, w.dtype, dev)
        self.q = torch.empty((self.T, h, w.d_nope + w.d_r), dtype=torch.bfloat16, device=dev)
        self.k_nope = torch.empty((self.T, h, w.d_nope), dtype=torch.bfloat16, device=dev)
        self.v = torch.empty((self.T, h, w.d_v), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((self.T, h, w.d_v), dtype=out_dtype, device=dev)
        self.lse = torch.empty((self.T, h), dtype=torch.float32, device=dev)
        ws = max(C.mla_linear_workspace_bytes(self.T, w.d_c, h * w.d_nope),
                 C.mla_linear_workspace_bytes(self.T, w.d_c, h * w.d_v))
        self.ws = torch.empty(max(1, ws // 4), dtype=torch.float32, device=dev)
        torch.cuda.synchronize(dev)

    def keys_values(self, stream=None):
        w = self.w
        C.mla_linear(self.c, self.dw.w_uk.view(-1, w.d_c), self.k_nope.view(self.T, -1), self.ws,
                     stream)
        C.mla_linear(self.c, self.dw.w_uv.view(-1, w.d_c), self.v.view(self.T, -1), self.ws,
                     stream)

    def query(self, stream=None):
        C.mla_prefill_query(self.q_nope, self.q_rope, self.cu, self.max_len, self.q,
                            rope_theta=self.w.theta, stream=stream)

    def attend(self, stream=None):
        C.mla_prefill_fwd(self.q, self.k_nope, self.k_rope, self.v, self.cu, self.max_len,
                          self.out, self.lse, dev_status=self.dw.status, stream=stream)

    def run(self, stream=None):
        self.keys_values(stream)
        self.query(stream)
        self.attend(stream)
        return self.out

    def attention_flops(self) -> float:
        """Causal attention flops: 2 (192 + 128) per (query, visible key) pair per head."""
        pairs = float(sum(int(L) * (int(L) + 1) // 2 for L in self.lens_np))
        w = self.w
        return 2.0 * (w.d_nope + w.d_r + w.d_v) * pairs * w.h
