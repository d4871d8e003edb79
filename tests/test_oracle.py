"""Pins for the fp64 oracle against things other than itself.

Each test checks the oracle against the numbers printed on the pages, a
closed form, an independent restatement (complex-number RoPE, a 50-digit
mpmath brute force written with scalar loops), or an invariant of the
mathematics. ``test_mutants_are_caught`` plants plausible mistakes in the
oracle (on the CPU) and checks that these pins reject every one of them.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as O
from mla_latent_kv_03_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")


def golden(key):
    with open(GOLDEN) as f:
        return json.load(f)[key]["value"]


# ---------------------------------------------------------------------------
# Closed forms printed on the pages
# ---------------------------------------------------------------------------

def test_bytes_per_token_match_pages():
    assert O.latent_bytes_per_token() == golden("latent_bytes_per_token_layer")
    assert O.gqa_bytes_per_token() == golden("gqa_bytes_per_token_layer")
    assert O.naive_bytes_per_token() == golden("naive_bytes_per_token_layer")
    gqa = O.gqa_bytes_per_token()
    assert 100.0 * O.latent_bytes_per_token() / gqa == golden("latent_vs_gqa_percent")
    assert 100.0 * O.naive_bytes_per_token() / gqa == golden("naive_vs_gqa_percent")
    saving = 100.0 * (1 - O.latent_bytes_per_token() / O.naive_bytes_per_token())
    assert saving == golden("latent_saving_vs_naive_percent")


def test_whole_model_cache_and_concurrency_match_pages():
    mb = O.cache_bytes(O.gqa_bytes_per_token(), 28, 1024) / 1e6
    assert math.floor(mb) == golden("gqa_28_layers_1024_tokens_MB_floor")
    # Reading: 32 GiB and DeepSeek-V2-Lite's 27 layers for both layouts.
    gib32 = 32 * 2 ** 30
    g = O.max_concurrency(gib32, 1024, O.gqa_bytes_per_token(), 27)
    m = O.max_concurrency(gib32, 1024, O.latent_bytes_per_token(), 27)
    assert g == golden("concurrency_32GB_seq1024_gqa")
    assert m == golden("concurrency_32GB_seq1024_mla")
    assert round(m / g, 2) == golden("concurrency_ratio")


def _crossover(state_bytes, per_token_bytes):
    return math.ceil(state_bytes / per_token_bytes)


def test_hybrid_crossovers_match_pages():
    # Qwen3-Next-80B-A3B: GDN 16 key heads, 32 value heads, dims 128, conv 4;
    # standard attention GQA with 2 KV heads of 256.
    s = O.hybrid_state_bytes(32, 128, 128) + O.hybrid_conv_bytes(128, 16, 128, 32, 4)
    assert _crossover(s, O.hybrid_gqa_bytes(1, 2, 256)) == golden("crossover_tokens_qwen3_next_gqa")
    # Kimi-Linear-48B-A3B: KDA 32 heads of 128, conv 4; MLA 512 + 64.
    s = O.hybrid_state_bytes(32, 128, 128) + O.hybrid_conv_bytes(128, 32, 128, 32, 4)
    assert _crossover(s, O.hybrid_mla_bytes(1)) == golden("crossover_tokens_kimi_linear_mla")
    # The hybrid page's MLA formula is the same 1,152 B/token as the other page's.
    assert O.hybrid_mla_bytes(1) == O.latent_bytes_per_token()


def test_serving_pool_bytes():
    # B=64 x 4096 tokens x 1,152 B: the latent cache one decode step reads.
    assert W.latent_cache_bytes_for([4096] * 64) == 301_989_888


# ---------------------------------------------------------------------------
# RoPE: independent restatement as complex multiplication, and invariants
# ---------------------------------------------------------------------------

def _rope_complex(x, pos, base):
    d = x.shape[-1]
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    theta = np.array([base ** (-(2.0 * i) / d) for i in range(half)])
    r = z * np.exp(1j * np.asarray(pos, float).reshape(-1, *([1] * (x.ndim - 1))) * theta)
    return np.concatenate([r.real, r.imag], axis=-1)


def test_rope_equals_complex_rotation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((9, 3, 64))
    pos = np.array([0, 1, 2, 7, 100, 1023, 4095, 20000, 32767])
    # fp64 angle rounding grows with the angle: ~pos * 2^-52 absolute
    np.testing.assert_allclose(O.rope(x, pos, 10000.0), _rope_complex(x, pos, 10000.0),
                               rtol=0, atol=3e-11)


def test_rope_invariants():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 64))
    k = rng.standard_normal((1, 64))
    # position 0 is the identity
    np.testing.assert_array_equal(O.rope(q, [0], 10000.0), q)
    # norm preserved
    for p in (1, 17, 4096):
        assert abs(np.linalg.norm(O.rope(q, [p], 1e4)) - np.linalg.norm(q)) < 1e-12
    # <R(m) q, R(n) k> depends only on m - n
    d1 = float(np.sum(O.rope(q, [130], 1e4) * O.rope(k, [100], 1e4)))
    d2 = float(np.sum(O.rope(q, [30], 1e4) * O.rope(k, [0], 1e4)))
    assert abs(d1 - d2) < 1e-10
    # pair 0 has inverse frequency 1: position pi/2 is not an integer, but
    # position 1 rotates pair 0 by exactly one radian
    e = np.zeros((1, 64)); e[0, 0] = 1.0
    r = O.rope(e, [1], 1e4)
    assert abs(r[0, 0] - math.cos(1.0)) < 1e-15 and abs(r[0, 32] - math.sin(1.0)) < 1e-15


# ---------------------------------------------------------------------------
# RMSNorm invariants
# ---------------------------------------------------------------------------

def test_rmsnorm_invariants():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 512)) * np.array([[0.1], [1], [3], [10], [1e-3]])
    eps = 1e-6
    y = O.rms_norm(x, np.ones(512), eps)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-12)
    # direction is unchanged (positive rescale of each row)
    cos = np.sum(x * y, -1) / np.linalg.norm(x, axis=-1) / np.linalg.norm(y, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=0, atol=1e-12)
    # the weight multiplies elementwise
    w = rng.standard_normal(512)
    np.testing.assert_allclose(O.rms_norm(x, w, eps), y * w, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------
# 50-digit brute force on tiny inputs (scalar loops, complex-number RoPE,
# softmax without max subtraction): an independent statement of the naive
# form of the mini-infer-17 page, section "版本 1: MLAAttentionNaive".
# ---------------------------------------------------------------------------

mp = pytest.importorskip("mpmath")


def _brute_force(c_raw, kpe_raw, kv_pos, q_nope, q_pe, q_pos, Wuk, Wuv, w, eps,
                 base, scale):
    mp.mp.dps = 50
    f = lambda v: mp.mpf(float(v))  # noqa: E731
    L, C = c_raw.shape
    n, H, D = q_nope.shape
    Vd = Wuv.shape[2]

    def norm_row(x):
        ms = mp.fsum(f(v) ** 2 for v in x) / len(x)
        inv = 1 / mp.sqrt(ms + f(eps))
        return [f(v) * inv * f(wi) for v, wi in zip(x, w)]

    def rot(x, p):
        half = len(x) // 2
        out = [None] * len(x)
        for i in range(half):
            z = mp.mpc(f(x[i]), f(x[i + half])) * mp.expj(f(p) * mp.power(f(base), -mp.mpf(2 * i) / len(x)))
            out[i], out[i + half] = z.real, z.imag
        return out

    chat = [norm_row(c_raw[t]) for t in range(L)]
    krot = [rot(kpe_raw[t], kv_pos[t]) for t in range(L)]
    out = np.zeros((n, H, Vd))
    lse = np.zeros((n, H))
    for i in range(n):
        for h in range(H):
            qr = rot(q_pe[i, h], q_pos[i])
            scores = []
            vis = [t for t in range(L) if t <= q_pos[i]]
            for t in vis:
                acc = mp.mpf(0)
                for d in range(D):
                    knope = mp.fsum(chat[t][c] * f(Wuk[h, c, d]) for c in range(C))
                    acc += f(q_nope[i, h, d]) * knope
                for r in range(len(qr)):
                    acc += qr[r] * krot[t][r]
                scores.append(f(scale) * acc)
            z = mp.fsum(mp.exp(s) for s in scores)
            lse[i, h] = float(mp.log(z))
            for v in range(Vd):
                tot = mp.mpf(0)
                for t, s in zip(vis, scores):
                    vt = mp.fsum(chat[t][c] * f(Wuv[h, c, v]) for c in range(C))
                    tot += mp.exp(s) / z * vt
                out[i, h, v] = float(tot)
    return out, lse


def _tiny_case(seed=7, L=5, q=3, H=2, C=8, R=4, D=4, Vd=4):
    rng = np.random.default_rng(seed)
    c_raw = rng.standard_normal((L, C)) * 2.0
    kpe_raw = rng.standard_normal((L, R))
    kv_pos = np.arange(L)
    q_nope = rng.standard_normal((q, H, D))
    q_pe = rng.standard_normal((q, H, R))
    q_pos = np.arange(L - q, L)
    Wuk = rng.standard_normal((H, C, D)) / math.sqrt(C)
    Wuv = rng.standard_normal((H, C, Vd)) / math.sqrt(C)
    w = 1.0 + 0.5 * rng.standard_normal(C)
    return dict(c_kv_raw=c_raw, k_pe_raw=kpe_raw, kv_positions=kv_pos, q_nope=q_nope,
                q_pe=q_pe, q_positions=q_pos, W_uk=Wuk, W_uv=Wuv, rms_weight=w,
                eps=1e-6, base=10000.0, scale=1.0 / math.sqrt(D + R))


def _check_against_brute_force(case):
    args = (case["c_kv_raw"], case["k_pe_raw"], case["kv_positions"], case["q_nope"],
            case["q_pe"], case["q_positions"], case["W_uk"], case["W_uv"],
            case["rms_weight"], case["eps"], case["base"], case["scale"])
    bf_out, bf_lse = _brute_force(*args)
    naive = O.mla_sequence_naive(*args)
    absorbed, _, lse = O.mla_sequence_absorbed(*args)
    # the full key/value cache form: expanded rows, then plain attention
    c_hat = O.rms_norm(case["c_kv_raw"], case["rms_weight"], case["eps"])
    k_rot = O.rope(case["k_pe_raw"], case["kv_positions"], case["base"])
    rows = O.naive_kv_rows(c_hat, k_rot, case["W_uk"], case["W_uv"])
    q = np.concatenate([case["q_nope"], O.rope(case["q_pe"], case["q_positions"], case["base"])], -1)
    expanded = O.expanded_attention(rows, q, case["q_positions"], case["scale"],
                                    nope_dim=case["q_nope"].shape[-1],
                                    rope_dim=case["q_pe"].shape[-1])
    return (max(float(np.max(np.abs(naive - bf_out))), float(np.max(np.abs(expanded - bf_out)))),
            float(np.max(np.abs(absorbed - bf_out))), float(np.max(np.abs(lse - bf_lse))))


@pytest.mark.parametrize("seed", [7, 8])
def test_oracle_matches_50_digit_brute_force(seed):
    e_naive, e_abs, e_lse = _check_against_brute_force(_tiny_case(seed))
    assert e_naive < 1e-13 and e_abs < 1e-13 and e_lse < 1e-13, (e_naive, e_abs, e_lse)


def test_naive_rows_are_the_pages_10240_bytes():
    """mini-infer-17, "版本 1": 16 x (192 + 128) x 2 = 10,240 bytes/token/layer."""
    rng = np.random.default_rng(3)
    rows = O.naive_kv_rows(rng.standard_normal((2, 512)), rng.standard_normal((2, 64)),
                           rng.standard_normal((16, 512, 128)), rng.standard_normal((16, 512, 128)))
    assert rows.shape == (2, 16, 320)
    assert rows.shape[1] * rows.shape[2] * 2 == golden("naive_bytes_per_token_layer")
    # every head carries the same shared rope key
    assert np.array_equal(rows[:, 0, 128:192], rows[:, 15, 128:192])


# ---------------------------------------------------------------------------
# Algebraic identity and invariants at the real head sizes
# ---------------------------------------------------------------------------

def _seq_case(seed, L, q, H=16):
    rng = np.random.default_rng(seed)
    return dict(
        c_kv_raw=rng.standard_normal((L, 512)), k_pe_raw=rng.standard_normal((L, 64)),
        kv_positions=np.arange(L), q_nope=rng.standard_normal((q, H, 128)),
        q_pe=rng.standard_normal((q, H, 64)), q_positions=np.arange(L - q, L),
        W_uk=rng.standard_normal((H, 512, 128)) / math.sqrt(512),
        W_uv=rng.standard_normal((H, 512, 128)) / math.sqrt(512),
        rms_weight=np.ones(512), eps=1e-6, base=10000.0, scale=1.0 / math.sqrt(192))


def _args(c):
    return (c["c_kv_raw"], c["k_pe_raw"], c["kv_positions"], c["q_nope"], c["q_pe"],
            c["q_positions"], c["W_uk"], c["W_uv"], c["rms_weight"], c["eps"],
            c["base"], c["scale"])


def test_absorbed_equals_naive():
    """mini-infer-17, section "版本 3": the absorbed form is the same math."""
    c = _seq_case(11, L=300, q=4)
    naive = O.mla_sequence_naive(*_args(c))
    absorbed, _, _ = O.mla_sequence_absorbed(*_args(c))
    rel = np.linalg.norm(absorbed - naive) / np.linalg.norm(naive)
    assert rel < 1e-12
    # far inside the page's fp32 bar of 1e-4
    assert np.max(np.abs(absorbed - naive)) < golden("absorbed_vs_naive_fp32_max_abs_bound") * 1e-6


def test_softmax_weights_sum_to_one():
    """Latent part all ones: the output is the sum of the softmax weights."""
    c = _seq_case(12, L=70, q=6)
    rows = O.latent_cache_rows(c["c_kv_raw"], c["k_pe_raw"], c["kv_positions"],
                               c["rms_weight"], c["eps"], c["base"])
    rows[:, :512] = 1.0
    q_abs = O.absorb_q(c["q_nope"], c["q_pe"], c["q_positions"], c["W_uk"], c["base"])
    o, lse = O.latent_attention(q_abs, rows, c["q_positions"], c["scale"])
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)
    assert np.all(np.isfinite(lse))


def test_single_token_returns_its_value():
    c = _seq_case(13, L=1, q=1)
    out = O.mla_sequence_naive(*_args(c))
    chat = O.rms_norm(c["c_kv_raw"], c["rms_weight"], c["eps"])
    v = np.einsum("c,hcv->hv", chat[0], c["W_uv"])
    np.testing.assert_allclose(out[0], v, rtol=1e-13, atol=1e-15)


def test_equal_rows_return_that_value():
    c = _seq_case(14, L=40, q=2)
    c["c_kv_raw"][:] = c["c_kv_raw"][0]
    c["k_pe_raw"][:] = 0.0     # identical keys at every position
    out = O.mla_sequence_naive(*_args(c))
    chat = O.rms_norm(c["c_kv_raw"][:1], c["rms_weight"], c["eps"])[0]
    v = np.einsum("c,hcv->hv", chat, c["W_uv"])
    np.testing.assert_allclose(out, np.broadcast_to(v, out.shape), rtol=1e-12, atol=1e-14)


def test_prefill_row_equals_decode_of_its_prefix():
    """Causal rows: query row j of a chunk equals a decode over kv 0..pos_j."""
    c = _seq_case(15, L=90, q=20)
    full = O.mla_sequence_naive(*_args(c))
    for j in (0, 7, 19):
        p = int(c["q_positions"][j])
        d = dict(c)
        d["c_kv_raw"], d["k_pe_raw"] = c["c_kv_raw"][:p + 1], c["k_pe_raw"][:p + 1]
        d["kv_positions"] = c["kv_positions"][:p + 1]
        d["q_nope"], d["q_pe"] = c["q_nope"][j:j + 1], c["q_pe"][j:j + 1]
        d["q_positions"] = c["q_positions"][j:j + 1]
        np.testing.assert_allclose(O.mla_sequence_naive(*_args(d))[0], full[j],
                                   rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("cuts", [[0, 100], [0, 1, 100], [0, 37, 38, 64, 100], [0, 0, 50, 100, 100]])
def test_merge_of_any_partition_equals_whole(cuts):
    c = _seq_case(16, L=100, q=1)
    rows = O.latent_cache_rows(c["c_kv_raw"], c["k_pe_raw"], c["kv_positions"],
                               c["rms_weight"], c["eps"], c["base"])
    q_abs = O.absorb_q(c["q_nope"], c["q_pe"], c["q_positions"], c["W_uk"], c["base"])
    o_all, lse_all = O.latent_attention(q_abs, rows, c["q_positions"], c["scale"])
    parts, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        # a part sees tokens [a, b): shift positions so the causal test is kept
        o, l = O.latent_attention(q_abs, rows[a:b], c["q_positions"] - a, c["scale"])
        parts.append(o); lses.append(l)
    o, l = O.merge_partials(np.stack(parts), np.stack(lses))
    np.testing.assert_allclose(o, o_all, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, lse_all, rtol=1e-13)


def test_empty_sequence_gives_zero():
    c = _seq_case(17, L=0, q=0)
    o, lse = O.latent_attention(np.zeros((1, 16, 576)), np.zeros((0, 576)), np.array([-1]), 0.1)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    o, lse = O.merge_partials(np.zeros((2, 1, 16, 512)), np.full((2, 1, 16), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    del c


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_dropping_rmsnorm_or_rope_breaks_parity():
    """The two mistakes the mini-infer-17 page reports (pitfall 3: no
    kv_a_layernorm, max diff 0.165; the RoPE-less naive version, 0.2655) must
    move the output far beyond the bf16 tolerance (rel-L2 5e-3)."""
    c = _seq_case(18, L=200, q=2)
    c["c_kv_raw"] = c["c_kv_raw"] * 3.0   # a latent whose RMS is not 1
    ref = O.mla_sequence_naive(*_args(c))
    no_norm = O.naive_attention(c["c_kv_raw"], O.rope(c["k_pe_raw"], c["kv_positions"], 1e4),
                                c["q_nope"], O.rope(c["q_pe"], c["q_positions"], 1e4),
                                c["W_uk"], c["W_uv"], c["q_positions"], c["scale"])
    no_rope = O.naive_attention(O.rms_norm(c["c_kv_raw"], 1.0, 1e-6), c["k_pe_raw"], c["q_nope"],
                                c["q_pe"], c["W_uk"], c["W_uv"], c["q_positions"], c["scale"])
    assert _rel(no_norm, ref) > 0.5
    assert _rel(no_rope, ref) > 0.1


def test_paged_gather_reads_what_slot_mapping_wrote():
    w = W.make("paged", [7, 33, 64, 65, 0, 1], [1, 1, 1, 1, 0, 1], 16, 16, "f32", seed=3, extra_blocks=5)
    rows = np.arange(w.num_tokens, dtype=np.float64)[:, None] * np.ones((1, 4))
    cache = np.full((w.num_blocks, 16, 4), np.nan)
    flat = cache.reshape(-1, 4)
    flat[w.slot_mapping] = rows                      # scatter, as the cache write does
    for b in range(w.batch):
        got = O.gather_paged(cache, w.block_table[b], int(w.seq_lens[b]), 16)
        np.testing.assert_array_equal(got, rows[w.token_range(b)])
    # every written slot is distinct, so no token overwrites another
    assert len(set(w.slot_mapping.tolist())) == w.num_tokens


# ---------------------------------------------------------------------------
# Planted mistakes: each plausible error in the oracle must fail a pin above.
# ---------------------------------------------------------------------------

def _rope_interleaved(x, positions, base):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    pos = np.asarray(positions, np.float64).reshape((-1,) + (1,) * (x.ndim - 1))
    ang = pos * O.rope_inv_freq(d, base)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * np.cos(ang) - b * np.sin(ang)
    out[..., 1::2] = b * np.cos(ang) + a * np.sin(ang)
    return out


_ROPE = O.rope


def _rope_sign_flipped(x, positions, base):
    return _ROPE(x, -np.asarray(positions), base)


def _rms_no_eps_sum(x, weight, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) * np.asarray(weight, np.float64)


def _absorb_heads_swapped(q_nope, q_pe, q_positions, W_uk, base):
    return np.concatenate([np.einsum("hcd,nhd->nhc", np.asarray(W_uk)[::-1], q_nope),
                           _ROPE(q_pe, q_positions, base)], -1)


def _visible_off_by_one(q_positions, kv_len):
    t = np.arange(kv_len)
    return t[None, :] < np.asarray(q_positions)[:, None]


def _naive_rows_value_from_uk(c_hat, k_rot, W_uk, W_uv):
    c_hat, k_rot = np.asarray(c_hat, np.float64), np.asarray(k_rot, np.float64)
    L, H = c_hat.shape[0], np.asarray(W_uk).shape[0]
    k = np.einsum("tc,hcd->thd", c_hat, W_uk)
    return np.concatenate([k, np.broadcast_to(k_rot[:, None, :], (L, H, k_rot.shape[-1])), k], -1)


MUTANTS = {
    "naive_rows_value_from_W_uk": ("naive_kv_rows", _naive_rows_value_from_uk),
    "rope_interleaved_pairs": ("rope", _rope_interleaved),
    "rope_wrong_direction": ("rope", _rope_sign_flipped),
    "rmsnorm_sum_not_mean": ("rms_norm", _rms_no_eps_sum),
    "absorb_wrong_head": ("absorb_q", _absorb_heads_swapped),
    "causal_off_by_one": ("causal_visible", _visible_off_by_one),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutants_are_caught(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(O, name, fn)
    caught = []
    try:
        e_naive, e_abs, e_lse = _check_against_brute_force(_tiny_case(7))
        caught.append(max(e_naive, e_abs, e_lse) > 1e-6)
    except Exception:
        caught.append(True)
    if name == "rope":
        rng = np.random.default_rng(0)
        x = rng.standard_normal((4, 2, 64))
        pos = np.array([0, 3, 50, 1000])
        caught.append(not np.allclose(O.rope(x, pos, 1e4), _rope_complex(x, pos, 1e4)))
    assert any(caught), f"planted mistake {mutant} passed every pin"


# ---------------------------------------------------------------------------
# FP8 (e4m3) cache rows
# ---------------------------------------------------------------------------

def test_e4m3_every_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert int((~finite).sum()) == 2                      # S.1111.111
    assert np.nanmax(vals) == O.E4M3_MAX and np.nanmin(vals) == -O.E4M3_MAX
    assert np.array_equal(O.e4m3_encode(vals[finite]), codes[finite])
    assert np.array_equal(O.e4m3_round(vals[finite]), vals[finite])


def test_e4m3_round_matches_torch_float8_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (0.01, 0.3, 3.0, 60.0)])
    x = np.clip(x, -O.E4M3_MAX, O.E4M3_MAX).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(x), ref)


def test_e4m3_ties_go_to_even_and_large_values_saturate():
    # 1.0625 lies halfway between 1.0 (mantissa 0) and 1.125 (mantissa 1)
    assert O.e4m3_round(1.0625) == 1.0 and O.e4m3_round(1.1875) == 1.25
    assert O.e4m3_round(-2.0 ** -10) == 0.0                # half the smallest subnormal
    assert O.e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8       # 1.5 subnormal steps -> 2
    assert O.e4m3_round(1e6) == O.E4M3_MAX and O.e4m3_round(-500.0) == -O.E4M3_MAX


def test_fp8_rows_dequantise_within_half_a_step():
    rng = np.random.default_rng(12)
    c = rng.standard_normal((40, 512))
    k_pe = rng.standard_normal((40, 64))
    codes, k_rot = O.fp8_latent_rows(c, k_pe, np.arange(40), np.ones(512), 1e-6, 1e4, 0.05)
    c_hat = O.rms_norm(c, np.ones(512), 1e-6)
    deq = O.e4m3_decode(codes) * 0.05
    # half a step of a 3-bit mantissa (relative 2^-4), or half the subnormal step
    bound = np.maximum(np.abs(c_hat) * 2.0 ** -4, 0.05 * 2.0 ** -10) + 1e-15
    assert np.all(np.abs(deq - c_hat) <= bound)
    # and a plain rounding would not be enough: the error is that of e4m3, not bf16
    assert np.max(np.abs(deq - c_hat)) > 2.0 ** -9
    assert np.array_equal(k_rot, O.rope(k_pe, np.arange(40), 1e4))


# ---------------------------------------------------------------------------
# Projections either side of the attention. With one-hot weights a projection
# only moves inputs, so the layout the page states (q_proj viewed per head as
# [qk_nope | qk_rope] then split; the kv_a output split at kv_lora_rank; o_proj
# over the heads' values laid head after head) is checked entry by entry.
# ---------------------------------------------------------------------------

def _one_hot(rows, cols, rng):
    src = rng.permutation(cols)[:rows]
    Wt = np.zeros((rows, cols))
    Wt[np.arange(rows), src] = 1.0
    return Wt, src


def test_q_proj_one_hot_weights_pick_head_major_nope_then_rope():
    rng = np.random.default_rng(21)
    H, D = 3, 640
    W_q, src = _one_hot(H * 192, D, rng)
    x = rng.standard_normal((4, D))
    q_nope, q_pe = O.q_proj(x, W_q, H)
    assert q_nope.shape == (4, H, 128) and q_pe.shape == (4, H, 64)
    for t in range(4):
        for h in range(H):
            for d in range(128):
                assert q_nope[t, h, d] == x[t, src[h * 192 + d]]
            for d in range(64):
                assert q_pe[t, h, d] == x[t, src[h * 192 + 128 + d]]


def test_kv_a_proj_one_hot_weights_split_latent_then_rope_key():
    rng = np.random.default_rng(22)
    D = 704
    W, src = _one_hot(576, D, rng)
    x = rng.standard_normal((3, D))
    c_kv, k_pe = O.kv_a_proj(x, W)
    assert c_kv.shape == (3, 512) and k_pe.shape == (3, 64)
    for t in range(3):
        assert all(c_kv[t, c] == x[t, src[c]] for c in range(512))
        assert all(k_pe[t, d] == x[t, src[512 + d]] for d in range(64))


def test_o_proj_one_hot_weights_read_heads_in_order():
    rng = np.random.default_rng(23)
    H, D = 2, 192
    W_o, src = _one_hot(D, H * 128, rng)
    a = rng.standard_normal((5, H, 128))
    y = O.o_proj(a, W_o)
    for t in range(5):
        for j in range(D):
            h, v = divmod(int(src[j]), 128)
            assert y[t, j] == a[t, h, v]


def test_projections_are_linear_in_the_weight_rows():
    # a weight row that is the sum of two one-hot rows adds the two inputs
    rng = np.random.default_rng(24)
    D = 256
    x = rng.standard_normal((2, D))
    W = np.zeros((576, D))
    W[7, 3] = 1.0
    W[7, 11] = 2.0
    W[600 - 30, 5] = -1.0
    c_kv, k_pe = O.kv_a_proj(x, W)
    assert np.allclose(c_kv[:, 7], x[:, 3] + 2 * x[:, 11], rtol=0, atol=1e-15)
    assert np.allclose(k_pe[:, 570 - 512], -x[:, 5], rtol=0, atol=1e-15)


def test_layer_naive_equals_absorbed_and_is_causal():
    rng = np.random.default_rng(25)
    H, D, T, new = 2, 256, 9, 3
    hid = rng.standard_normal((T, D))
    s = 1 / math.sqrt(D)
    W_q = rng.standard_normal((H * 192, D)) * s
    W_kv_a = rng.standard_normal((576, D)) * s
    W_uk = rng.standard_normal((H, 512, 128)) / math.sqrt(512)
    W_uv = rng.standard_normal((H, 512, 128)) / math.sqrt(512)
    W_o = rng.standard_normal((D, H * 128)) / math.sqrt(H * 128)
    pos = np.arange(T)
    args = (W_q, W_kv_a, W_uk, W_uv, W_o, np.ones(512), 1e-6, 1e4, 1 / math.sqrt(192))
    y = O.mla_layer_naive(hid, pos, *args, num_new=new)
    # the same layer through the absorbed form
    q_nope, q_pe = O.q_proj(hid[-new:], W_q, H)
    c_kv, k_pe = O.kv_a_proj(hid, W_kv_a)
    out, _, _ = O.mla_sequence_absorbed(c_kv, k_pe, pos, q_nope, q_pe, pos[-new:], W_uk, W_uv,
                                        np.ones(512), 1e-6, 1e4, 1 / math.sqrt(192))
    assert np.allclose(y, O.o_proj(out, W_o), rtol=1e-12, atol=1e-12)
    # query row j sees tokens up to its own position: dropping later tokens
    # leaves it unchanged
    y_short = O.mla_layer_naive(hid[:T - 1], pos[:T - 1], *args, num_new=new - 1)
    assert np.allclose(y[:new - 1], y_short, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Interleaved RoPE pairing (the option the pages leave open)
# ---------------------------------------------------------------------------

def test_interleaved_rope_is_complex_rotation_of_adjacent_pairs():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((5, 3, 64))
    pos = np.array([0, 1, 7, 100, 4095])
    got = O.rope(x, pos, 1e4, interleaved=True)
    inv = 1e4 ** (-np.arange(32) * 2 / 64)
    for t in range(5):
        z = (x[t, :, 0::2] + 1j * x[t, :, 1::2]) * np.exp(1j * pos[t] * inv)
        assert np.allclose(got[t, :, 0::2], z.real, rtol=0, atol=1e-12)
        assert np.allclose(got[t, :, 1::2], z.imag, rtol=0, atol=1e-12)
    assert np.array_equal(O.rope(x, np.zeros(5, int), 1e4, interleaved=True), x)


def test_interleaved_rope_is_rotate_half_on_permuted_coordinates():
    # moving element 2i to i and 2i+1 to 32 + i turns one pairing into the other
    rng = np.random.default_rng(32)
    x = rng.standard_normal((6, 64))
    pos = rng.integers(0, 5000, 6)
    perm = np.concatenate([np.arange(0, 64, 2), np.arange(1, 64, 2)])
    inter = O.rope(x, pos, 1e4, interleaved=True)
    half = O.rope(x[:, perm], pos, 1e4)
    assert np.allclose(inter[:, perm], half, rtol=0, atol=1e-12)
    # and the two pairings differ as functions (the option is not a no-op)
    assert not np.allclose(inter, O.rope(x, pos, 1e4), atol=1e-3)


def test_interleaved_attention_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(33)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    s = [O.rope(q[None], [m], 1e4, True)[0] @ O.rope(k[None], [n], 1e4, True)[0]
         for m, n in ((10, 3), (110, 103), (1010, 1003))]
    assert np.allclose(s, s[0], rtol=0, atol=1e-9)
