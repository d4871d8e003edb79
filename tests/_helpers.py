"""Glue between workloads, the oracle and device tensors (test code only)."""

import numpy as np

from oracle import mla_oracle as O

# Parity bars: bf16 I/O max abs <= 2e-2 and rel-L2 <= 5e-3; fp32 I/O max abs
# <= 1e-4 (the mini-infer-17 page's own bar for the absorbed form).
BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 5e-3
F32_MAX_ABS = 1e-4


def to_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def ref_out(w, seqs=None, heads=None):
    """Naive-form oracle output [num_q, H', 128] for the chosen sequences and
    heads (rows of other sequences are left as NaN)."""
    heads = np.arange(w.num_heads) if heads is None else np.asarray(heads)
    seqs = range(w.batch) if seqs is None else seqs
    out = np.full((w.num_q, len(heads), 128), np.nan)
    for b in seqs:
        tr, qr = w.token_range(b), w.q_range(b)
        if qr.stop == qr.start:
            continue
        out[qr] = O.mla_sequence_naive(
            w.c_kv_raw[tr], w.k_pe_raw[tr], w.kv_positions[tr], w.q_nope[qr][:, heads],
            w.q_pe[qr][:, heads], w.q_positions[qr], w.W_uk[heads], w.W_uv[heads],
            w.rms_weight, w.rms_eps, w.rope_base, w.softmax_scale)
    return out


def ref_cache_rows(w):
    return O.latent_cache_rows(w.c_kv_raw, w.k_pe_raw, w.kv_positions, w.rms_weight,
                               w.rms_eps, w.rope_base)


def ref_q_abs(w):
    return O.absorb_q(w.q_nope, w.q_pe, w.q_positions, w.W_uk, w.rope_base)


def ref_o_lat_from(w, cache_np, q_abs_np, seqs=None):
    """Latent-attention oracle on the GPU's own cache rows and q_abs (isolates
    the decode + combine kernels)."""
    o = np.full((w.num_q, w.num_heads, 512), np.nan)
    for b in (range(w.batch) if seqs is None else seqs):
        qr = w.q_range(b)
        if qr.stop == qr.start:
            continue
        rows = O.gather_paged(cache_np, w.block_table[b], int(w.seq_lens[b]), w.block_size)
        o[qr], _ = O.latent_attention(q_abs_np[qr], rows, w.q_positions[qr], w.softmax_scale)
    return o


def errors(got, ref):
    m = ~np.isnan(ref)
    d = got[m] - ref[m]
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    nrm = float(np.linalg.norm(ref[m]))
    rel = float(np.linalg.norm(d) / nrm) if nrm > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_close(got, ref, dtype, what=""):
    max_abs, rel = errors(got, ref)
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"{what}: max abs {max_abs:.3g} > {F32_MAX_ABS}"
    else:
        assert max_abs <= BF16_MAX_ABS, f"{what}: max abs {max_abs:.3g} > {BF16_MAX_ABS}"
        assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3g} > {BF16_REL_L2}"
    return max_abs, rel


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def ref_out_absorbed(w, seqs, rows_of=None):
    """Output [num_q, H, 128] through the oracle's absorbed form (cache rows,
    q_abs, latent attention, W_uv), which the oracle's tests hold equal to the
    naive form to 1e-12; cheap enough for every head of long sequences.
    rows_of(b) may pick a subset of sequence b's query rows (indices into
    w.q_range(b)); other rows stay NaN."""
    out = np.full((w.num_q, w.num_heads, 128), np.nan)
    for b in seqs:
        tr, qr = w.token_range(b), w.q_range(b)
        if qr.stop == qr.start:
            continue
        idx = np.arange(qr.start, qr.stop)
        if rows_of is not None:
            idx = idx[np.asarray(rows_of(b), dtype=np.int64)]
        rows = O.latent_cache_rows(w.c_kv_raw[tr], w.k_pe_raw[tr], w.kv_positions[tr],
                                   w.rms_weight, w.rms_eps, w.rope_base)
        q_abs = O.absorb_q(w.q_nope[idx], w.q_pe[idx], w.q_positions[idx], w.W_uk, w.rope_base)
        o_lat, _ = O.latent_attention(q_abs, rows, w.q_positions[idx], w.softmax_scale)
        out[idx] = O.out_proj(o_lat, w.W_uv)
    return out
