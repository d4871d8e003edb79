"""Plain fp64 CPU oracle for MLA latent-KV paged decode.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it. It imports nothing from the CUDA library
or its Python binding, and the library shares no code with it.

Everything is written in float64 NumPy, in the order the sources state it,
with no blocking, fusion or reordering. Inputs stored as bf16 or fp32 are
upcast exactly to fp64 before use.

Sources (web pages; section headings as printed on them)
--------------------------------------------------------
[MI17]  "mini-infer-17: MLA Attention -- from KV-cache compression to matrix
        absorption" (smarter.xin): sections "MLA 的数学结构" (math structure),
        "版本 1: MLAAttentionNaive", "版本 2: MLAAttentionLatentCache",
        "版本 3: MLAAttentionAbsorbed (矩阵吸收)", "踩坑记录" (pitfalls 2 and 3),
        "实验结果" (results tables), "设计取舍" (design choices).
[VLB07] "07. MLA / Mamba / MoE in vLLM source" (vLLM learning book):
        sections 2.1 "算法核心", 2.2 "vLLM 源码挂载点", 2.3 "与 KV manager 的接缝",
        2.4 "Decoupled RoPE", self-check question 1.
[HYB]   bxzpzcl.cn article on KV/state-cache management for hybrid (GDN/KDA)
        models in vLLM/SGLang: sections 2.2 and 2.3 (cache-size formulas).

Readings where the sources are silent:
  * RoPE uses rotate-half pairing (x_i, x_{i+d/2}), inv_freq_i = base^(-2i/d).
  * A token's RoPE position is its 0-based index within its sequence.
  * The latent cache stores the RMSNorm'd c_kv (the pages' engine stores the
    raw latent and norms it at attention time; the two are the same math).
  * Query row j of a sequence with L cached tokens (new ones included) and
    q_len new query rows sits at position L - q_len + j and sees kv 0..pos.
  * A query row that sees no token gives a zero output and lse = -inf.

Every function below is pinned by tests in ``tests/test_oracle.py`` against
something other than itself (closed forms printed on the pages, a complex-
number restatement of RoPE, a 50-digit mpmath brute force, invariants).
"""

from __future__ import annotations

import numpy as np

KV_LORA_RANK = 512      # [MI17 "MLA 的数学结构"]: kv_lora_rank = 512
QK_ROPE_HEAD_DIM = 64   # [MI17 "MLA 的数学结构"]: qk_rope_head_dim = 64
QK_NOPE_HEAD_DIM = 128  # [VLB07 self-check 1]: qk_nope_head_dim 128
V_HEAD_DIM = 128        # [MI17 "版本 1"]: 16 x (192 + 128) -> v_head_dim 128


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Per-token transforms
# ---------------------------------------------------------------------------

def rms_norm(x, weight, eps: float) -> np.ndarray:
    """kv_a_layernorm applied to the compressed latent.

    y = x / sqrt(mean(x^2) + eps) * weight over the last axis.
    [MI17 "版本 1": kv_b_proj(kv_a_layernorm(compressed_kv));
     pitfall 3: the latent must be normed before it meets W_uk/W_uv.]
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(weight)


def rope_inv_freq(rope_dim: int, base: float) -> np.ndarray:
    """inv_freq_i = base^(-2i/rope_dim), i < rope_dim/2 (standard RoPE).

    [VLB07 2.4 "Decoupled RoPE"; MI17 "MLA 的数学结构": K_pe = x W_kr + RoPE]
    """
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return np.float64(base) ** (-2.0 * i / rope_dim)


def rope(x, positions, base: float, interleaved: bool = False) -> np.ndarray:
    """RoPE on the last axis of ``x``.

    ``x`` is [T, ..., d]; ``positions`` is [T]. Pair i is rotated by angle
    positions[t] * inv_freq_i: the pair (x_i, x_{i+d/2}) (rotate-half, the
    reading taken for the pages) or, with ``interleaved``, (x_{2i}, x_{2i+1})
    (the other pairing in use, left open by the pages).
    [VLB07 2.4; MI17 "MLA 的数学结构" (k_pe shared by all heads, MQA style)]
    """
    x = _f64(x)
    d = x.shape[-1]
    half = d // 2
    pos = _f64(positions).reshape((-1,) + (1,) * (x.ndim - 1))
    ang = pos * rope_inv_freq(d, base)           # [T, 1.., half]
    cos, sin = np.cos(ang), np.sin(ang)
    if interleaved:
        x1, x2 = x[..., 0::2], x[..., 1::2]
        out = np.empty_like(x)
        out[..., 0::2] = x1 * cos - x2 * sin
        out[..., 1::2] = x2 * cos + x1 * sin
        return out
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def latent_cache_rows(c_kv_raw, k_pe_raw, positions, rms_weight, eps: float,
                      base: float, interleaved: bool = False) -> np.ndarray:
    """The row that the paged cache must hold for each token: [c_hat || k_hat].

    c_hat = RMSNorm(c_kv_raw) * w (512), k_hat = RoPE(k_pe_raw, pos) (64).
    [VLB07 2.3: MLA cache shape (n_blocks, block, 1, latent_d + rope_d);
     VLB07 2.2: write c_kv to the KV cache by slot_mapping;
     MI17 "版本 2": the cache holds only compressed_kv + k_pe]
    """
    return np.concatenate(
        [rms_norm(c_kv_raw, rms_weight, eps), rope(k_pe_raw, positions, base, interleaved)],
        axis=-1)


# ---------------------------------------------------------------------------
# Absorbed form: the per-step decode path
# ---------------------------------------------------------------------------

def absorb_q(q_nope, q_pe, q_positions, W_uk, base: float,
             interleaved: bool = False) -> np.ndarray:
    """q_abs[n,h] = [W_uk[h] @ q_nope[n,h] || RoPE(q_pe[n,h], pos_n)].

    W_uk is [H, kv_lora_rank, qk_nope] (the absorbed key weight of
    [MI17 "版本 3" _build_absorbed]: kv_b_proj.weight viewed per head, nope
    rows, transposed). q_lat[n,h,c] = sum_d W_uk[h,c,d] * q_nope[n,h,d].
    """
    q_lat = np.einsum("hcd,nhd->nhc", _f64(W_uk), _f64(q_nope))
    return np.concatenate([q_lat, rope(q_pe, q_positions, base, interleaved)], axis=-1)


def causal_visible(q_positions, kv_len: int) -> np.ndarray:
    """mask[n, t] = True where query n may attend kv token t (t <= pos_n).

    [MI17 pitfall 2: causal mask = triu(ones, diagonal=1) filled with -inf]
    """
    t = np.arange(kv_len)
    return t[None, :] <= np.asarray(q_positions)[:, None]


def latent_attention(q_abs, kv_rows, q_positions, scale: float,
                     kv_lora_rank: int = KV_LORA_RANK):
    """Scores and softmax-weighted sum directly against the latent rows.

    q_abs [n, H, 576], kv_rows [L, 576] (one sequence), q_positions [n].
    s[n,h,t] = scale * q_abs[n,h] . kv_rows[t]   (nope and rope terms in one
    dot product: [MI17 "设计取舍": the two score parts are summed, then a
    hand-written softmax); causal mask; p = softmax_t(s);
    o_lat[n,h] = sum_t p[n,h,t] * kv_rows[t, :kv_lora_rank].
    Returns (o_lat [n,H,512], lse [n,H]) with lse = log sum_t exp(s) (natural
    log). Rows that see no token return zeros and lse = -inf.
    """
    q_abs = _f64(q_abs)
    kv_rows = _f64(kv_rows)
    n, H, _ = q_abs.shape
    L = kv_rows.shape[0]
    o = np.zeros((n, H, kv_lora_rank))
    lse = np.full((n, H), -np.inf)
    if L == 0 or n == 0:
        return o, lse
    s = scale * np.einsum("nhk,tk->nht", q_abs, kv_rows)
    vis = causal_visible(q_positions, L)[:, None, :]           # [n,1,L]
    s = np.where(vis, s, -np.inf)
    any_vis = vis.any(axis=-1)                                  # [n,1]
    m = np.where(any_vis, s.max(axis=-1), 0.0)                  # [n,H]
    p = np.where(vis, np.exp(s - m[..., None]), 0.0)
    denom = p.sum(axis=-1)
    ok = denom > 0
    safe = np.where(ok, denom, 1.0)
    o = np.einsum("nht,tc->nhc", p / safe[..., None], kv_rows[:, :kv_lora_rank])
    o = np.where(ok[..., None], o, 0.0)
    lse = np.where(ok, m + np.log(safe), -np.inf)
    return o, lse


def merge_partials(o_parts, lse_parts):
    """Combine split-KV partial results (flash-decoding merge).

    o_parts [S, ...,  D] are the normalised partial outputs of disjoint token
    subsets, lse_parts [S, ...] their log-sum-exp (natural log, -inf = empty).
    o = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M), M = max_s lse_s;
    lse = M + log sum_s exp(lse_s - M). This is the softmax identity over a
    partition of the tokens; the pages do not print it.
    """
    o_parts = _f64(o_parts)
    lse_parts = _f64(lse_parts)
    M = lse_parts.max(axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - Ms), 0.0)
    den = w.sum(axis=0)
    safe = np.where(den > 0, den, 1.0)
    o = (w[..., None] * o_parts).sum(axis=0) / safe[..., None]
    o = np.where((den > 0)[..., None], o, 0.0)
    lse = np.where(den > 0, Ms + np.log(safe), -np.inf)
    return o, lse


def out_proj(o_lat, W_uv) -> np.ndarray:
    """out[n,h,v] = sum_c o_lat[n,h,c] * W_uv[h,c,v].

    W_uv is [H, kv_lora_rank, v_head_dim] ([MI17 "版本 3" _build_absorbed]:
    the value rows of kv_b_proj.weight per head, transposed).
    """
    return np.einsum("nhc,hcv->nhv", _f64(o_lat), _f64(W_uv))


# ---------------------------------------------------------------------------
# Naive (expanded) form: the end-to-end reference
# ---------------------------------------------------------------------------

def naive_attention(c_hat, k_rot, q_nope, q_rot, W_uk, W_uv, q_positions,
                    scale: float) -> np.ndarray:
    """[MI17 "版本 1: MLAAttentionNaive"]: expand K and V per head, then attend.

    c_hat [L, 512] normed latent, k_rot [L, 64] RoPE'd shared key,
    q_nope [n, H, 128], q_rot [n, H, 64] RoPE'd query rope part.
    K_nope[t,h] = c_hat[t] @ W_uk[h]   ([MI17 "MLA 的数学结构": K_nope = C_KV W_uk])
    V[t,h]      = c_hat[t] @ W_uv[h]   (V = C_KV W_uv)
    K[t,h]      = [K_nope[t,h] || k_rot[t]]   (k_pe shared by every head)
    Q[n,h]      = [q_nope[n,h] || q_rot[n,h]]
    out[n,h]    = softmax_t(scale * Q.K, causal) @ V   -> [n, H, 128]
    """
    c_hat, k_rot = _f64(c_hat), _f64(k_rot)
    q_nope, q_rot = _f64(q_nope), _f64(q_rot)
    W_uk, W_uv = _f64(W_uk), _f64(W_uv)
    L = c_hat.shape[0]
    n, H, _ = q_nope.shape
    dv = W_uv.shape[-1]
    out = np.zeros((n, H, dv))
    if L == 0 or n == 0:
        return out
    k_nope = np.einsum("tc,hcd->thd", c_hat, W_uk)               # [L,H,128]
    v = np.einsum("tc,hcv->thv", c_hat, W_uv)                    # [L,H,128]
    K = np.concatenate(
        [k_nope, np.broadcast_to(k_rot[:, None, :], (L, H, k_rot.shape[-1]))],
        axis=-1)                                                 # [L,H,192]
    Q = np.concatenate([q_nope, q_rot], axis=-1)                 # [n,H,192]
    s = scale * np.einsum("nhe,the->nht", Q, K)
    vis = causal_visible(q_positions, L)[:, None, :]
    s = np.where(vis, s, -np.inf)
    any_vis = vis.any(axis=-1)
    m = np.where(any_vis, s.max(axis=-1), 0.0)
    p = np.where(vis, np.exp(s - m[..., None]), 0.0)
    den = p.sum(axis=-1)
    safe = np.where(den > 0, den, 1.0)
    out = np.einsum("nht,thv->nhv", p / safe[..., None], v)
    return np.where((den > 0)[..., None], out, 0.0)


# ---------------------------------------------------------------------------
# FP8 latent cache. The pages name "FP8 KV" handling of MLA only as a later
# chapter ([MI17] "下一章": 量化对 MLA / MoE 的特殊处理); the reading taken here
# (stated as such): each row holds c_hat / kv_scale as OCP e4m3 codes (1 sign,
# 4 exponent bits with bias 7, 3 mantissa bits, no infinities, 448 the largest
# finite value), rounded to nearest with ties to even and saturated at +-448,
# followed by k_rot in bf16; kv_scale is one positive number per cache.
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 code (NaN for S.1111.111)."""
    c = np.asarray(codes, np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return sign * val


def e4m3_round(x) -> np.ndarray:
    """x rounded to the e4m3 grid: nearest value, ties to the even mantissa,
    saturated at +-448. In the binade [2^e, 2^(e+1)) (and the subnormals,
    which share the spacing of e = -6) the grid is k * 2^(e-3), k integer, and
    k is even exactly when the mantissa is."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
    step = np.exp2(e - 3)
    q = a / step
    k = np.floor(q)
    frac = q - k
    k = np.where(frac > 0.5, k + 1, np.where(frac < 0.5, k, k + (k % 2)))
    v = np.minimum(k * step, E4M3_MAX)
    return np.copysign(np.where(a > 0, v, 0.0), x)


def e4m3_encode(v) -> np.ndarray:
    """Code of each value already on the e4m3 grid (|v| <= 448)."""
    v = np.asarray(v, np.float64)
    sign = (np.signbit(v)).astype(np.int64) << 7
    a = np.abs(v)
    sub = a < 2.0 ** -6
    e = np.floor(np.log2(np.where(sub, 1.0, a)))
    m_norm = np.round((a / np.exp2(e) - 1.0) * 8.0).astype(np.int64)
    m_sub = np.round(a / 2.0 ** -9).astype(np.int64)
    code = np.where(sub, m_sub, ((e.astype(np.int64) + 7) << 3) | m_norm)
    return (sign | code).astype(np.uint8)


def fp8_latent_rows(c_kv_raw, k_pe_raw, positions, rms_weight, eps: float, base: float,
                    kv_scale: float, interleaved: bool = False):
    """The FP8 cache row of each token (reading above): the e4m3 codes of
    c_hat / kv_scale [T, 512] uint8, and k_rot [T, 64] (stored in bf16).
    Dequantised latent = e4m3_decode(codes) * kv_scale."""
    c_hat = rms_norm(c_kv_raw, rms_weight, eps)
    codes = e4m3_encode(e4m3_round(c_hat / float(kv_scale)))
    return codes, rope(k_pe_raw, positions, base, interleaved)


def naive_kv_rows(c_hat, k_rot, W_uk, W_uv) -> np.ndarray:
    """[MI17 "版本 1: MLAAttentionNaive"]: the rows the full key/value cache holds.

    For token t and head h: [K_nope[t,h] (128) || k_rot[t] (64) || V[t,h] (128)]
    with K_nope[t,h] = c_hat[t] @ W_uk[h] and V[t,h] = c_hat[t] @ W_uv[h]: the
    page caches the whole key (nope || rope) and the value of every head, 16 x
    (192 + 128) x 2 = 10,240 bytes/token/layer in bf16. "版本 2" re-expands the
    latent cache into exactly these rows at every step.  -> [L, H, 320]
    """
    c_hat, k_rot = _f64(c_hat), _f64(k_rot)
    W_uk, W_uv = _f64(W_uk), _f64(W_uv)
    L, H = c_hat.shape[0], W_uk.shape[0]
    k_nope = np.einsum("tc,hcd->thd", c_hat, W_uk)
    v = np.einsum("tc,hcv->thv", c_hat, W_uv)
    rope_part = np.broadcast_to(k_rot[:, None, :], (L, H, k_rot.shape[-1]))
    return np.concatenate([k_nope, rope_part, v], axis=-1)


def expanded_attention(kv_rows, q, q_positions, scale: float,
                       nope_dim: int = QK_NOPE_HEAD_DIM,
                       rope_dim: int = QK_ROPE_HEAD_DIM) -> np.ndarray:
    """The naive form's attention step over expanded rows ([MI17 "版本 1"]).

    kv_rows [L, H, nope+rope+v] = [K_nope || k_rot || V] per head (as
    naive_kv_rows), q [n, H, nope+rope] = [q_nope || q_rot];
    out[n,h] = softmax_t(scale * q[n,h] . K[t,h], causal) @ V[t,h] -> [n, H, v].
    """
    kv_rows, q = _f64(kv_rows), _f64(q)
    kd = nope_dim + rope_dim
    K, V = kv_rows[..., :kd], kv_rows[..., kd:]
    n, H = q.shape[0], q.shape[1]
    L = kv_rows.shape[0]
    out = np.zeros((n, H, V.shape[-1]))
    if L == 0 or n == 0:
        return out
    s = scale * np.einsum("nhe,the->nht", q, K)
    vis = causal_visible(q_positions, L)[:, None, :]
    s = np.where(vis, s, -np.inf)
    any_vis = vis.any(axis=-1)
    m = np.where(any_vis, s.max(axis=-1), 0.0)
    p = np.where(vis, np.exp(s - m[..., None]), 0.0)
    den = p.sum(axis=-1)
    safe = np.where(den > 0, den, 1.0)
    out = np.einsum("nht,thv->nhv", p / safe[..., None], V)
    return np.where((den > 0)[..., None], out, 0.0)


def mla_sequence_naive(c_kv_raw, k_pe_raw, kv_positions, q_nope, q_pe,
                       q_positions, W_uk, W_uv, rms_weight, eps: float,
                       base: float, scale: float, interleaved: bool = False) -> np.ndarray:
    """End-to-end attention output for one sequence from raw inputs.

    kv_a_layernorm on the latent, RoPE on k_pe and q_pe, then the naive form.
    [MI17 "版本 1" and pitfall 3; VLB07 2.2 forward steps 1-4]
    """
    c_hat = rms_norm(c_kv_raw, rms_weight, eps)
    k_rot = rope(k_pe_raw, kv_positions, base, interleaved)
    q_rot = rope(q_pe, q_positions, base, interleaved)
    return naive_attention(c_hat, k_rot, q_nope, q_rot, W_uk, W_uv,
                           q_positions, scale)


def mla_sequence_absorbed(c_kv_raw, k_pe_raw, kv_positions, q_nope, q_pe,
                          q_positions, W_uk, W_uv, rms_weight, eps: float,
                          base: float, scale: float):
    """The same output through the absorbed form (cache rows, q_abs, latent
    attention, W_uv). [MI17 "版本 3"]. Returns (out, o_lat, lse)."""
    rows = latent_cache_rows(c_kv_raw, k_pe_raw, kv_positions, rms_weight,
                             eps, base)
    q_abs = absorb_q(q_nope, q_pe, q_positions, W_uk, base)
    o_lat, lse = latent_attention(q_abs, rows, q_positions, scale,
                                  kv_lora_rank=_f64(W_uk).shape[1])
    return out_proj(o_lat, W_uv), o_lat, lse


# ---------------------------------------------------------------------------
# Projections either side of the attention ([MI17] "版本 1: MLAAttentionNaive":
# q_proj, kv_a_proj_with_mqa, o_proj; [VLB07] 2.2). Weights are in a linear
# layer's [out, in] layout: y = x W^T.
# ---------------------------------------------------------------------------

def q_proj(hidden, W_q, num_heads: int):
    """q = hidden W_q^T viewed per head as [qk_nope | qk_rope] and split:
    returns (q_nope [T, H, 128], q_pe [T, H, 64])."""
    q = _f64(hidden) @ _f64(W_q).T
    q = q.reshape(q.shape[0], num_heads, QK_NOPE_HEAD_DIM + QK_ROPE_HEAD_DIM)
    return q[..., :QK_NOPE_HEAD_DIM], q[..., QK_NOPE_HEAD_DIM:]


def kv_a_proj(hidden, W_kv_a):
    """kv_a_proj_with_mqa: hidden W_kv_a^T split into the latent and the
    shared rope key: returns (c_kv [T, 512], k_pe [T, 64]), both raw (the
    kv_a_layernorm and RoPE come after, in the cache write)."""
    kv = _f64(hidden) @ _f64(W_kv_a).T
    return kv[:, :KV_LORA_RANK], kv[:, KV_LORA_RANK:]


def o_proj(attn_out, W_o):
    """o_proj over the heads' concatenated values: attn_out [T, H, 128]
    flattened to [T, H * 128], times W_o^T -> [T, hidden]."""
    a = _f64(attn_out)
    return a.reshape(a.shape[0], -1) @ _f64(W_o).T


def mla_layer_naive(hidden, kv_positions, W_q, W_kv_a, W_uk, W_uv, W_o, rms_weight,
                    eps: float, base: float, scale: float, num_new: int) -> np.ndarray:
    """One sequence through the whole attention layer in the naive form: the
    sequence's hidden states (all of its tokens, the last num_new of them
    being the step's queries) projected to queries and to latents, the naive
    attention, o_proj. Returns [num_new, hidden]. [MI17] "版本 1"."""
    q_nope, q_pe = q_proj(hidden[-num_new:], W_q, _f64(W_uk).shape[0])
    c_kv, k_pe = kv_a_proj(hidden, W_kv_a)
    q_positions = np.asarray(kv_positions)[-num_new:]
    out = mla_sequence_naive(c_kv, k_pe, kv_positions, q_nope, q_pe, q_positions, W_uk, W_uv,
                             rms_weight, eps, base, scale)
    return o_proj(out, W_o)


def gather_paged(cache, block_table_row, seq_len: int, block_size: int):
    """Read one sequence's rows back out of a paged cache, in logical order.

    cache [n_blocks, block_size, row]; logical token t lives in physical block
    block_table_row[t // block_size] at offset t % block_size
    ([VLB07 2.3 and the PagedAttention block-table indirection]).
    """
    cache = np.asarray(cache)
    t = np.arange(seq_len)
    blocks = np.asarray(block_table_row)[t // block_size]
    return cache[blocks, t % block_size]


# ---------------------------------------------------------------------------
# Cache-size closed forms (bytes)
# ---------------------------------------------------------------------------

def latent_bytes_per_token(kv_lora_rank=KV_LORA_RANK,
                           rope_dim=QK_ROPE_HEAD_DIM, elem_bytes=2) -> int:
    """[MI17 "MLA 的数学结构" and "版本 2"]: (512 + 64) x 2 = 1,152 B/token/layer."""
    return (kv_lora_rank + rope_dim) * elem_bytes


def naive_bytes_per_token(num_heads=16, qk_nope=QK_NOPE_HEAD_DIM,
                          qk_rope=QK_ROPE_HEAD_DIM, v_dim=V_HEAD_DIM,
                          elem_bytes=2) -> int:
    """[MI17 "版本 1"]: full K (192) + V (128) per head: 16 x 320 x 2 = 10,240."""
    return num_heads * (qk_nope + qk_rope + v_dim) * elem_bytes


def gqa_bytes_per_token(kv_heads=4, head_dim=128, elem_bytes=2) -> int:
    """[MI17 background]: 4 KV heads x 128 x 2 (K+V) x 2 B = 2,048."""
    return kv_heads * head_dim * 2 * elem_bytes


def cache_bytes(bytes_per_token_layer: int, num_layers: int, tokens: int) -> int:
    """Whole-model cache bytes: per-token-per-layer size x layers x tokens."""
    return bytes_per_token_layer * num_layers * tokens


def max_concurrency(memory_bytes: int, seq_len: int, bytes_per_token_layer: int,
                    num_layers: int) -> int:
    """How many sequences of ``seq_len`` tokens fit in ``memory_bytes``."""
    return memory_bytes // (seq_len * bytes_per_token_layer * num_layers)


def hybrid_mla_bytes(seq_len, kv_lora_rank=KV_LORA_RANK,
                     rope_dim=QK_ROPE_HEAD_DIM) -> int:
    """[HYB 2.3]: MLA := 2 * seq_len * (kv_lora_rank + qk_rope_head_dim)."""
    return 2 * seq_len * (kv_lora_rank + rope_dim)


def hybrid_gqa_bytes(seq_len, kv_heads, head_dim, tp=1) -> float:
    """[HYB 2.3]: GQA := 2 * 2 * seq_len * num_key_value_heads * head_dim / TP."""
    return 2 * 2 * seq_len * kv_heads * head_dim / tp


def hybrid_state_bytes(num_v_heads, head_k_dim, head_v_dim, tp=1) -> float:
    """[HYB 2.3]: S := 2 * num_v_heads / TP * head_k_dim * head_v_dim."""
    return 2 * num_v_heads / tp * head_k_dim * head_v_dim


def hybrid_conv_bytes(head_k_dim, num_k_heads, head_v_dim, num_v_heads,
                      conv_kernel, tp=1) -> float:
    """[HYB 2.3]: Conv := 2 * (head_k_dim*num_k_heads*2 + head_v_dim*num_v_heads)
    / TP * (conv_kernel_size - 1)."""
    return (2 * (head_k_dim * num_k_heads * 2 + head_v_dim * num_v_heads) / tp
            * (conv_kernel - 1))
