"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds data generation only (random draws, bf16 rounding of the
stored values, block tables, slot mappings, query layouts). It contains none
of the attention arithmetic, so the oracle and the CUDA path stay independent.

Input recipe (every workload):
  * q_nope, q_pe, c_kv_raw, k_pe_raw ~ N(0, 1);
  * W_uk, W_uv ~ N(0, 1/512) (variance 1/512), shape [H, 512, 128];
  * RMSNorm weight 1, eps 1e-6, RoPE base 10000, softmax scale 1/sqrt(192);
  * values drawn in fp32 and rounded (round-to-nearest-even) to the storage
    dtype, so the oracle and the GPU see bit-identical inputs;
  * the physical block pool is a seeded random permutation of exactly the
    blocks the sequences need (plus ``extra_blocks`` spare ones), assigned in
    logical order; unused block-table entries are -1;
  * ``seq_lens`` include the new tokens; query row j of a sequence with
    ``q_len`` rows sits at position seq_len - q_len + j.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

KV_LORA_RANK = 512
ROPE_DIM = 64
NOPE_DIM = 128
V_DIM = 128
ROW = KV_LORA_RANK + ROPE_DIM


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even); return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 array of the values the storage dtype can hold exactly."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(bf16_bits(x))
    if dtype == "f32":
        return x
    raise ValueError(dtype)


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                      # "f32" or "bf16": storage of every tensor
    num_heads: int
    block_size: int
    seq_lens: np.ndarray            # int32 [B]
    q_lens: np.ndarray              # int32 [B]
    num_blocks: int
    block_table: np.ndarray         # int32 [B, max_blocks], -1 padded
    # per token of every sequence, sequence-major, positions 0..L-1
    c_kv_raw: np.ndarray            # f32 [T, 512] (values exact in dtype)
    k_pe_raw: np.ndarray            # f32 [T, 64]
    kv_positions: np.ndarray        # int32 [T]
    slot_mapping: np.ndarray        # int64 [T]
    token_seq: np.ndarray           # int32 [T]
    is_new: np.ndarray              # bool  [T]: written by this step
    # queries
    query_start_loc: np.ndarray     # int32 [B+1]
    q_nope: np.ndarray              # f32 [Nq, H, 128]
    q_pe: np.ndarray                # f32 [Nq, H, 64]
    q_positions: np.ndarray         # int32 [Nq]
    # weights
    W_uk: np.ndarray                # f32 [H, 512, 128]
    W_uv: np.ndarray                # f32 [H, 512, 128]
    rms_weight: np.ndarray          # f32 [512]
    rms_eps: float = 1e-6
    rope_base: float = 10000.0
    softmax_scale: float = 1.0 / math.sqrt(NOPE_DIM + ROPE_DIM)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_q(self) -> int:
        return int(self.q_nope.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.kv_positions.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def token_range(self, b: int) -> slice:
        start = int(np.sum(self.seq_lens[:b]))
        return slice(start, start + int(self.seq_lens[b]))

    def q_range(self, b: int) -> slice:
        return slice(int(self.query_start_loc[b]), int(self.query_start_loc[b + 1]))

    def latent_bytes(self) -> int:
        """Bytes of latent cache the decode step reads (every visible row once)."""
        elem = 2 if self.dtype == "bf16" else 4
        return int(np.sum(self.seq_lens)) * ROW * elem


def make(name: str, seq_lens, q_lens, num_heads: int, block_size: int, dtype: str,
         seed: int, extra_blocks: int = 0) -> Workload:
    """Draw one workload. Draw order is fixed so a seed names a workload."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    assert seq_lens.shape == q_lens.shape and np.all(q_lens <= seq_lens)
    rng = np.random.default_rng(seed)
    H = num_heads
    B = seq_lens.shape[0]
    w_std = np.float32(1.0 / math.sqrt(KV_LORA_RANK))
    W_uk = rng.standard_normal((H, KV_LORA_RANK, NOPE_DIM), dtype=np.float32) * w_std
    W_uv = rng.standard_normal((H, KV_LORA_RANK, V_DIM), dtype=np.float32) * w_std
    Nq = int(q_lens.sum())
    q_nope = rng.standard_normal((Nq, H, NOPE_DIM), dtype=np.float32)
    q_pe = rng.standard_normal((Nq, H, ROPE_DIM), dtype=np.float32)
    T = int(seq_lens.sum())
    c_kv = rng.standard_normal((T, KV_LORA_RANK), dtype=np.float32)
    k_pe = rng.standard_normal((T, ROPE_DIM), dtype=np.float32)

    blocks_per_seq = [(int(L) + block_size - 1) // block_size for L in seq_lens]
    used = int(sum(blocks_per_seq))
    num_blocks = used + int(extra_blocks)
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(1, max(blocks_per_seq) if blocks_per_seq else 1)
    block_table = np.full((B, max_blocks), -1, dtype=np.int32)
    k = 0
    for b, nb in enumerate(blocks_per_seq):
        block_table[b, :nb] = perm[k:k + nb]
        k += nb

    kv_positions = np.concatenate(
        [np.arange(L, dtype=np.int32) for L in seq_lens]) if T else np.zeros(0, np.int32)
    token_seq = np.concatenate(
        [np.full(L, b, dtype=np.int32) for b, L in enumerate(seq_lens)]) if T else np.zeros(0, np.int32)
    bt = block_table[token_seq, kv_positions // block_size] if T else np.zeros(0, np.int32)
    slot_mapping = bt.astype(np.int64) * block_size + (kv_positions % block_size)
    is_new = kv_positions >= (seq_lens - q_lens)[token_seq] if T else np.zeros(0, bool)

    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    q_positions = np.concatenate(
        [np.arange(L - q, L, dtype=np.int32) for L, q in zip(seq_lens, q_lens)]) if Nq else np.zeros(0, np.int32)

    r = lambda a: round_to_dtype(a, dtype)  # noqa: E731
    return Workload(
        name=name, dtype=dtype, num_heads=H, block_size=block_size,
        seq_lens=seq_lens, q_lens=q_lens, num_blocks=num_blocks,
        block_table=block_table, c_kv_raw=r(c_kv), k_pe_raw=r(k_pe),
        kv_positions=kv_positions, slot_mapping=slot_mapping,
        token_seq=token_seq, is_new=is_new, query_start_loc=qsl,
        q_nope=r(q_nope), q_pe=r(q_pe), q_positions=q_positions,
        W_uk=r(W_uk), W_uv=r(W_uv),
        rms_weight=np.ones(KV_LORA_RANK, dtype=np.float32))


@dataclasses.dataclass
class LayerInputs:
    """Inputs of the projections either side of the attention for one
    workload: every token's hidden state (in the workload's token order) and
    the three weights in a linear layer's [out, in] layout."""
    hidden: np.ndarray   # f32 [T, D] (bf16 values)
    W_q: np.ndarray      # f32 [H * 192, D]
    W_kv_a: np.ndarray   # f32 [576, D]
    W_o: np.ndarray      # f32 [D, H * 128]


def layer_inputs(w: Workload, hidden_size: int = 2048, seed: int = 7) -> LayerInputs:
    """hidden ~ N(0, 1); W_q, W_kv_a ~ N(0, 1/D); W_o ~ N(0, 1/(H * 128));
    all rounded to bf16. D = 2048 is DeepSeek-V2-Lite's hidden size."""
    rng = np.random.default_rng(seed)
    H, D, T = w.num_heads, hidden_size, w.num_tokens
    s_in = np.float32(1.0 / math.sqrt(D))
    hidden = rng.standard_normal((T, D), dtype=np.float32)
    W_q = rng.standard_normal((H * (NOPE_DIM + ROPE_DIM), D), dtype=np.float32) * s_in
    W_kv_a = rng.standard_normal((KV_LORA_RANK + ROPE_DIM, D), dtype=np.float32) * s_in
    W_o = rng.standard_normal((D, H * V_DIM), dtype=np.float32) * np.float32(1.0 / math.sqrt(H * V_DIM))
    r = lambda a: round_to_dtype(a, "bf16")  # noqa: E731
    return LayerInputs(hidden=r(hidden), W_q=r(W_q), W_kv_a=r(W_kv_a), W_o=r(W_o))


# The workloads the pages' statement of the problem names, plus small cases of
# the same shapes that the oracle finishes in seconds.
def tiny(seed: int = 1) -> Workload:
    """B=2, 16 heads, seq_lens {7, 33}, block_size 16, fp32."""
    return make("tiny_fp32_B2_H16_L7-33_bs16", [7, 33], [1, 1], 16, 16, "f32", seed)


def v2lite(seq_len: int, seed: int = 2) -> Workload:
    """DeepSeek-V2-Lite-shaped single-layer decode: B=1, 16 heads, bf16, bs 64."""
    return make(f"v2lite_B1_H16_L{seq_len}_bf16", [seq_len], [1], 16, 64, "bf16", seed)


def serving(seed: int = 3, batch: int = 64, seq_len: int = 4096) -> Workload:
    """Serving-batch decode: B=64, every seq_len 4096, 16 heads, bf16, bs 64."""
    return make(f"serving_B{batch}_H16_L{seq_len}_bf16", [seq_len] * batch,
                [1] * batch, 16, 64, "bf16", seed)


def ragged_h128(seed: int = 4, batch: int = 32, max_len: int = 32768) -> Workload:
    """Many-head ragged decode: B=32, 128 heads, seq_len ~ U[1, 32768], bf16."""
    lens = np.random.default_rng(1000 + seed).integers(1, max_len + 1, size=batch)
    return make(f"ragged_B{batch}_H128_U1-{max_len}_bf16", lens, [1] * batch,
                128, 64, "bf16", seed)


def mixed(seed: int = 5, n_prefill: int = 4, cached: int = 2048, new: int = 512,
          n_decode: int = 60, decode_len: int = 1024, heads: int = 16) -> Workload:
    """Chunked prefill + decode: 4 x (2048 cached + 512 new causal rows) and
    60 decode sequences at seq_len 1024; 16 heads, bf16, bs 64."""
    lens = [cached + new] * n_prefill + [decode_len] * n_decode
    qs = [new] * n_prefill + [1] * n_decode
    return make(f"mixed_P{n_prefill}x{cached}+{new}_D{n_decode}x{decode_len}_H{heads}_bf16",
                lens, qs, heads, 64, "bf16", seed)


NAMED = {
    "tiny": tiny,
    "v2lite_1": lambda: v2lite(1),
    "v2lite_256": lambda: v2lite(256),
    "v2lite_1024": lambda: v2lite(1024),
    "serving": serving,
    "ragged_h128": ragged_h128,
    "mixed": mixed,
}


def by_name(name: str) -> Workload:
    return NAMED[name]()


def latent_cache_bytes_for(seq_lens, dtype: str = "bf16") -> int:
    elem = 2 if dtype == "bf16" else 4
    return int(np.sum(seq_lens)) * ROW * elem


def as_dict(w: Workload) -> Dict[str, object]:
    return dataclasses.asdict(w)


def describe(w: Workload) -> Dict[str, object]:
    return {"workload": w.name, "batch": w.batch, "num_heads": w.num_heads,
            "block_size": w.block_size, "dtype": w.dtype,
            "tokens": int(np.sum(w.seq_lens)), "num_q": w.num_q,
            "num_blocks": w.num_blocks}
