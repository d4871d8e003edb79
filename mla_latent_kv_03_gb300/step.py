"""Device buffers for one workload and the calls of one decode step.

`MlaDecodeStep` owns torch device tensors (torch is only the allocator and
stream provider here) and issues the libmla calls of one step:
  mla_cache_write (new tokens) -> mla_absorb_q -> mla_decode_paged
  -> mla_combine -> mla_out_proj.
"""

from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import libmla as L
from . import workloads as W
from .workloads import Workload


def _dev(a: np.ndarray, dtype, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


class MlaDecodeStep:
    def __init__(self, w: Workload, device: str = "cuda", num_ctas: int = 0,
                 cache_fill: Optional[float] = None, rope_interleaved: bool = False):
        self.w = w
        self.device = device
        self.cfg = L.make_config(w.num_heads, w.block_size, w.dtype, num_ctas=num_ctas,
                                 softmax_scale=w.softmax_scale, rms_eps=w.rms_eps,
                                 rope_base=w.rope_base, rope_interleaved=rope_interleaved)
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.dt = dt
        H = w.num_heads
        self.W_uk = _dev(w.W_uk, dt, device)
        self.W_uv = _dev(w.W_uv, dt, device)
        self.rms_weight = _dev(w.rms_weight, dt, device)
        self.block_table = _dev(w.block_table, torch.int32, device)
        self.seq_lens = _dev(w.seq_lens, torch.int32, device)
        self.query_start_loc = _dev(w.query_start_loc, torch.int32, device)
        self.q_nope = _dev(w.q_nope, dt, device)
        self.q_pe = _dev(w.q_pe, dt, device)
        self.q_positions = _dev(w.q_positions, torch.int32, device)
        # every token of every sequence (used to populate the cache)
        self.c_kv = _dev(w.c_kv_raw, dt, device)
        self.k_pe = _dev(w.k_pe_raw, dt, device)
        self.kv_positions = _dev(w.kv_positions, torch.int32, device)
        self.slot_mapping = _dev(w.slot_mapping, torch.int64, device)
        new = np.nonzero(w.is_new)[0]
        self.new_idx = new
        self.c_kv_new = self.c_kv[torch.from_numpy(new).to(device)].contiguous()
        self.k_pe_new = self.k_pe[torch.from_numpy(new).to(device)].contiguous()
        self.pos_new = self.kv_positions[torch.from_numpy(new).to(device)].contiguous()
        self.slot_new = self.slot_mapping[torch.from_numpy(new).to(device)].contiguous()
        self.cache = torch.empty((w.num_blocks, w.block_size, 576), dtype=dt, device=device)
        if cache_fill is not None:
            self.cache.fill_(cache_fill)
        Nq = w.num_q
        self.q_abs = torch.empty((Nq, H, 576), dtype=dt, device=device)
        self.o_lat = torch.empty((Nq, H, 512), dtype=torch.float32, device=device)
        self.out = torch.empty((Nq, H, 128), dtype=dt, device=device)
        ws_bytes = L.mla_decode_workspace_size(self.cfg, Nq, w.batch)
        if ws_bytes == 0:
            raise L.MlaError(L.MLA_OK + 2, "mla_decode_workspace_size")
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        L.mla_workspace_init(self.workspace)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    # -- cache population --------------------------------------------------
    def populate(self, include_new: bool = True) -> None:
        """Write every token (or every old token) into the paged cache."""
        if include_new:
            L.mla_cache_write(self.cfg, self.c_kv, self.k_pe, self.kv_positions,
                              self.slot_mapping, self.rms_weight, self.cache, self.status)
            return
        old = torch.from_numpy(np.nonzero(~self.w.is_new)[0]).to(self.device)
        if old.numel() == 0:
            return
        L.mla_cache_write(self.cfg, self.c_kv[old].contiguous(), self.k_pe[old].contiguous(),
                          self.kv_positions[old].contiguous(), self.slot_mapping[old].contiguous(),
                          self.rms_weight, self.cache, self.status)

    def write_new(self, stream=None) -> None:
        L.mla_cache_write(self.cfg, self.c_kv_new, self.k_pe_new, self.pos_new, self.slot_new,
                          self.rms_weight, self.cache, self.status, stream=stream)

    # -- one step ----------------------------------------------------------
    def absorb(self, stream=None) -> None:
        L.mla_absorb_q(self.cfg, self.q_nope, self.q_pe, self.q_positions, self.W_uk, self.q_abs,
                       stream=stream)

    def decode(self, stream=None) -> None:
        L.mla_decode_paged(self.cfg, self.q_abs, self.cache, self.block_table, self.seq_lens,
                           self.query_start_loc, self.workspace, stream=stream)

    def plan(self, stream=None) -> None:
        L.mla_decode_plan(self.cfg, self.seq_lens, self.query_start_loc, self.w.num_q,
                          self.block_table.shape[1], self.workspace, stream=stream)

    def decode_planned(self, stream=None) -> None:
        L.mla_decode_planned(self.cfg, self.q_abs, self.cache, self.block_table, self.w.batch,
                             self.workspace, stream=stream)

    def decode_combine(self, stream=None) -> None:
        L.mla_decode_combine(self.cfg, self.q_abs, self.cache, self.block_table, self.w.batch,
                             self.workspace, self.o_lat, stream=stream)

    def decode_paged_combine(self, stream=None) -> None:
        L.mla_decode_paged_combine(self.cfg, self.q_abs, self.cache, self.block_table,
                                   self.seq_lens, self.query_start_loc, self.workspace, self.o_lat,
                                   stream=stream)

    def combine(self, stream=None) -> None:
        L.mla_combine(self.cfg, self.workspace, self.w.batch, self.o_lat, stream=stream)

    def combine_out_proj(self, stream=None) -> None:
        L.mla_combine_out_proj(self.cfg, self.workspace, self.w.batch, self.w.num_q, self.W_uv,
                               self.out, stream=stream)

    def out_proj(self, stream=None) -> None:
        L.mla_out_proj(self.cfg, self.o_lat, self.W_uv, self.out, stream=stream)

    def step(self, write_new: bool = False, stream=None) -> torch.Tensor:
        if write_new:
            self.write_new(stream)
        self.absorb(stream)
        self.decode(stream)
        self.combine(stream)
        self.out_proj(stream)
        return self.out

    # -- the FP8 latent cache -----------------------------------------------
    def fp8_setup(self, kv_scale: float) -> None:
        """The FP8 cache ([num_blocks, block_size, 640] bytes) and its scale."""
        w = self.w
        self.kv_scale = float(kv_scale)
        self.cache8 = torch.empty((w.num_blocks, w.block_size, 640), dtype=torch.uint8,
                                  device=self.device)
        need = L.mla_decode_fp8_workspace_size(self.cfg, int(w.num_q), w.batch)
        if need == 0:
            raise L.MlaError(L.MLA_OK + 2, "mla_decode_fp8_workspace_size")
        if need > self.workspace.numel():
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
            L.mla_workspace_init(self.workspace)

    def fp8_populate(self) -> None:
        L.mla_cache_write_fp8(self.cfg, self.c_kv, self.k_pe, self.kv_positions,
                              self.slot_mapping, self.rms_weight, self.kv_scale, self.cache8,
                              self.status)

    def decode_paged_combine_fp8(self, stream=None) -> None:
        L.mla_decode_paged_combine_fp8(self.cfg, self.q_abs, self.cache8, self.block_table,
                                       self.seq_lens, self.query_start_loc, self.kv_scale,
                                       self.workspace, self.o_lat, stream=stream)

    # -- the projections either side (the whole attention layer) -----------
    def layer_setup(self, hidden_size: int = 2048, seed: int = 7) -> None:
        """Hidden states of every token and the q_proj / kv_a_proj / o_proj
        weights (bf16), plus the buffers the layer step writes."""
        w, dev = self.w, self.device
        li = W.layer_inputs(w, hidden_size, seed)
        self.layer = li
        self.hidden_size = hidden_size
        dt = torch.bfloat16
        self.hidden = _dev(li.hidden, dt, dev)
        self.W_q = _dev(li.W_q, dt, dev)
        self.W_kv_a = _dev(li.W_kv_a, dt, dev)
        self.W_o = _dev(li.W_o, dt, dev)
        new = torch.from_numpy(np.nonzero(w.is_new)[0]).to(dev)
        self.hidden_new = self.hidden[new].contiguous()
        self.y = torch.empty((w.num_q, hidden_size), dtype=dt, device=dev)
        # the split (and so the partials' size) depends on the token count
        need = min(L.mla_proj_workspace_size(self.cfg, max(n, 1), hidden_size)
                   for n in (w.num_tokens, w.num_q))
        need = max(L.mla_proj_workspace_size(self.cfg, max(n, 1), hidden_size)
                   for n in (w.num_tokens, w.num_q)) if need else 0
        if need == 0:
            raise L.MlaError(L.MLA_OK + 2, "mla_proj_workspace_size")
        self.proj_ws = torch.empty(need, dtype=torch.uint8, device=dev)
        L.mla_workspace_init(self.proj_ws)
        # a second projection workspace for kv_a_proj when it runs beside
        # q_proj (calls that share a workspace must not overlap)
        self.proj_ws_side = torch.empty(need, dtype=torch.uint8, device=dev)
        L.mla_workspace_init(self.proj_ws_side)
        self.ly_fork, self.ly_join = torch.cuda.Event(), torch.cuda.Event()

    def layer_populate(self) -> None:
        """kv_a_proj of every token, then the cache write of the old ones."""
        L.mla_kv_a_proj(self.cfg, self.hidden, self.W_kv_a, self.c_kv, self.k_pe, self.proj_ws)
        new = torch.from_numpy(np.nonzero(self.w.is_new)[0]).to(self.device)
        self.c_kv_new = self.c_kv[new].contiguous()
        self.k_pe_new = self.k_pe[new].contiguous()
        self.populate(include_new=False)

    def layer_step(self, stream=None, side=None) -> torch.Tensor:
        """One decode step of the whole layer: q_proj and kv_a_proj of the new
        tokens, their cache write, absorb, decode + merge, out_proj, o_proj.
        With a `side` stream, kv_a_proj and the cache write run there,
        concurrently with q_proj and the absorption on the current stream,
        and the decode waits for both."""
        if side is None:
            L.mla_q_proj(self.cfg, self.hidden_new, self.W_q, self.q_nope, self.q_pe, self.proj_ws,
                         stream=stream)
            L.mla_kv_a_proj(self.cfg, self.hidden_new, self.W_kv_a, self.c_kv_new, self.k_pe_new,
                            self.proj_ws, stream=stream)
            self.write_new(stream=stream)
            self.absorb(stream=stream)
        else:
            cur = torch.cuda.current_stream() if stream is None else stream
            self.ly_fork.record(cur)
            side.wait_event(self.ly_fork)
            with torch.cuda.stream(side):
                L.mla_kv_a_proj(self.cfg, self.hidden_new, self.W_kv_a, self.c_kv_new, self.k_pe_new,
                                self.proj_ws_side)
                self.write_new()
                self.ly_join.record(side)
            L.mla_q_proj(self.cfg, self.hidden_new, self.W_q, self.q_nope, self.q_pe, self.proj_ws,
                         stream=stream)
            self.absorb(stream=stream)
            cur.wait_event(self.ly_join)
        self.decode_paged_combine(stream=stream)
        self.out_proj(stream=stream)
        L.mla_o_proj(self.cfg, self.out, self.W_o, self.y, self.proj_ws, stream=stream)
        return self.y

    # -- the pages' other two forms (full K/V cache; latent re-expanded) ----
    def naive_setup(self) -> None:
        """Buffers of the expanded cache ([num_blocks, block_size, H, 320]) and
        the workspace of its calls."""
        w = self.w
        self.kv_naive = torch.empty((w.num_blocks, w.block_size, w.num_heads, 320),
                                    dtype=self.dt, device=self.device)
        n = L.mla_naive_workspace_size(self.cfg, w.num_q, self.block_table.shape[1],
                                       max(int(self.c_kv.shape[0]), 1))
        if n == 0:
            raise L.MlaError(L.MLA_OK + 2, "mla_naive_workspace_size")
        self.naive_ws = torch.empty(n, dtype=torch.uint8, device=self.device)
        L.mla_workspace_init(self.naive_ws)
        self.out_naive = torch.empty((w.num_q, w.num_heads, 128), dtype=self.dt, device=self.device)

    def naive_populate(self) -> None:
        """Version 1's cache: every token expanded into the rows of every head."""
        L.mla_naive_cache_write(self.cfg, self.c_kv, self.k_pe, self.kv_positions,
                                self.slot_mapping, self.rms_weight, self.W_uk, self.W_uv,
                                self.kv_naive, self.naive_ws)

    def naive_write_new(self, stream=None) -> None:
        """Version 1's cache write of the step's new tokens."""
        L.mla_naive_cache_write(self.cfg, self.c_kv_new, self.k_pe_new, self.pos_new,
                                self.slot_new, self.rms_weight, self.W_uk, self.W_uv,
                                self.kv_naive, self.naive_ws, stream=stream)

    def latent_expand(self, stream=None) -> None:
        """Version 2: re-expand the whole latent cache into kv_naive."""
        L.mla_latent_expand(self.cfg, self.cache, self.block_table, self.seq_lens, self.W_uk,
                            self.W_uv, self.kv_naive, self.naive_ws, stream=stream)

    def naive_decode(self, stream=None) -> None:
        L.mla_naive_decode(self.cfg, self.q_nope, self.q_pe, self.q_positions, self.kv_naive,
                           self.block_table, self.seq_lens, self.query_start_loc, self.naive_ws,
                           self.out_naive, stream=stream)

    def naive_prefill(self, stream=None) -> None:
        L.mla_naive_prefill(self.cfg, self.q_nope, self.q_pe, self.q_positions, self.kv_naive,
                            self.block_table, self.seq_lens, self.query_start_loc, self.naive_ws,
                            self.out_naive, stream=stream)

    # -- a prefill + decode batch split by form ----------------------------
    def hybrid_setup(self) -> None:
        """Prefill sequences (more than one new row) take the expanded form,
        decode sequences the absorbed one; the batch holds the prefill
        sequences first. Buffers of the expanded rows, the decode rows'
        query_start_loc from 0, and the fork/join events."""
        w = self.w
        ql = np.diff(w.query_start_loc)
        npf = int((ql > 1).sum())
        if not (np.all(ql[:npf] > 1) and np.all(ql[npf:] <= 1)):
            raise ValueError("hybrid step: prefill sequences must come first")
        self.hy_seqs = npf
        self.hy_rows = int(w.query_start_loc[npf])
        self.qsl_decode = _dev((w.query_start_loc[npf:] - w.query_start_loc[npf]).astype(np.int32),
                               torch.int32, self.device)
        self.naive_setup()
        self.hy_fork, self.hy_join = torch.cuda.Event(), torch.cuda.Event()

    def hybrid_prefill(self, stream=None) -> None:
        """The prefill sequences: their latent rows re-expanded per head, then
        the tensor-core attention of their rows."""
        P, R = self.hy_seqs, self.hy_rows
        L.mla_latent_expand(self.cfg, self.cache, self.block_table[:P], self.seq_lens[:P],
                            self.W_uk, self.W_uv, self.kv_naive, self.naive_ws, stream=stream)
        self.hybrid_prefill_attention(stream=stream)

    def hybrid_prefill_attention(self, stream=None) -> None:
        P, R = self.hy_seqs, self.hy_rows
        L.mla_naive_prefill(self.cfg, self.q_nope[:R], self.q_pe[:R], self.q_positions[:R],
                            self.kv_naive, self.block_table[:P], self.seq_lens[:P],
                            self.query_start_loc[:P + 1], self.naive_ws, self.out_naive[:R],
                            stream=stream)

    def hybrid_decode(self, stream=None) -> None:
        """The decode sequences through the absorbed step; their output rows go
        to out_naive as well."""
        P, R = self.hy_seqs, self.hy_rows
        L.mla_absorb_q(self.cfg, self.q_nope[R:], self.q_pe[R:], self.q_positions[R:], self.W_uk,
                       self.q_abs[R:], stream=stream)
        L.mla_decode_paged_combine(self.cfg, self.q_abs[R:], self.cache, self.block_table[P:],
                                   self.seq_lens[P:], self.qsl_decode, self.workspace,
                                   self.o_lat[R:], stream=stream)
        L.mla_out_proj(self.cfg, self.o_lat[R:], self.W_uv, self.out_naive[R:], stream=stream)

    def hybrid_step(self, side: torch.cuda.Stream) -> torch.Tensor:
        """The new tokens' latent rows, then the decode part on `side` and the
        prefill part on the current stream, concurrently."""
        self.write_new()
        cur = torch.cuda.current_stream()
        self.hy_fork.record(cur)
        side.wait_event(self.hy_fork)
        with torch.cuda.stream(side):
            self.hybrid_decode()
            self.hy_join.record(side)
        self.hybrid_prefill()
        cur.wait_event(self.hy_join)
        return self.out_naive

    def device_status(self):
        """(status, bits) of the decode workspace and of the cache-write word."""
        s1 = L.mla_get_device_status(self.workspace)
        s2 = L.mla_get_device_status(self.status)
        return s1, s2

    def decode_mode(self) -> int:
        """Kernel family the last plan chose: 0 = warp-mma tiles of 16 heads,
        1 = tensor-core tiles of 128 (row, head) rows. Synchronises."""
        return int(self.workspace[32:36].view(torch.int32).item())
