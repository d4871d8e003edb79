"""GPU parity of the projections either side of the attention (q_proj,
kv_a_proj_with_mqa, o_proj) and of the whole layer built from them, against
the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from _helpers import assert_close, bf16_ulp, to_f64
from mla_latent_kv_03_gb300 import libmla as L
from mla_latent_kv_03_gb300 import workloads as W
from mla_latent_kv_03_gb300.step import MlaDecodeStep
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    L.load()


def _bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))
    return torch.from_numpy(x).to(torch.bfloat16)


def _bound(x, Wt, ref):
    """One bf16 rounding of the fp32 result plus the fp32 summation error of
    any order over K terms (K * 2^-24 * sum |x_k w_k|)."""
    K = x.shape[1]
    mag = np.abs(to_f64(x)) @ np.abs(to_f64(Wt)).T
    return bf16_ulp(ref) + K * 2.0 ** -24 * mag


def _check(got, ref, bound, what):
    bad = ~(np.abs(got - ref) <= bound)
    if bad.any():
        idx = np.argwhere(bad)
        first = tuple(idx[0])
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} beyond the bound (NaN: {np.isnan(got).sum()}); "
            f"first at {first}: got {got[first]!r}, ref {ref[first]!r}, bound {bound[first]!r}; "
            f"bad rows {np.unique(idx[:, 0])[:8]}, bad last-index {np.unique(idx[:, -1])[:8]}")


def _ws(cfg, T, D):
    ws = torch.empty(L.mla_proj_workspace_size(cfg, T, D), dtype=torch.uint8, device=DEV)
    L.mla_workspace_init(ws)
    return ws


@pytest.mark.parametrize("T", [1, 7, 64, 300, 2108])
@pytest.mark.parametrize("H", [16, 128])
def test_q_proj_vs_oracle(T, H):
    D = 2048
    rng = np.random.default_rng(100 + T + H)
    cfg = L.make_config(H, 64, "bf16")
    x, Wq = _bf16(rng, (T, D)), _bf16(rng, (H * 192, D), D ** -0.5)
    q_nope = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    q_pe = torch.full((T, H, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg, T, D)
    L.mla_q_proj(cfg, x.to(DEV), Wq.to(DEV), q_nope, q_pe, ws)
    torch.cuda.synchronize()
    assert L.mla_get_device_status(ws)[0] == 0
    ref = to_f64(x) @ to_f64(Wq).T
    bound = _bound(x, Wq, ref).reshape(T, H, 192)
    rn, rp = O.q_proj(to_f64(x), to_f64(Wq), H)
    _check(to_f64(q_nope), rn, bound[..., :128], "q_nope")
    _check(to_f64(q_pe), rp, bound[..., 128:], "q_pe")


@pytest.mark.parametrize("T", [1, 5, 64, 129, 300, 2108])
def test_kv_a_proj_vs_oracle(T):
    D = 2048
    rng = np.random.default_rng(200 + T)
    cfg = L.make_config(16, 64, "bf16")
    x, Wkv = _bf16(rng, (T, D)), _bf16(rng, (576, D), D ** -0.5)
    c_kv = torch.full((T, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    k_pe = torch.full((T, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg, T, D)
    L.mla_kv_a_proj(cfg, x.to(DEV), Wkv.to(DEV), c_kv, k_pe, ws)
    torch.cuda.synchronize()
    assert L.mla_get_device_status(ws)[0] == 0
    ref = to_f64(x) @ to_f64(Wkv).T
    bound = _bound(x, Wkv, ref)
    rc, rk = O.kv_a_proj(to_f64(x), to_f64(Wkv))
    _check(to_f64(c_kv), rc, bound[:, :512], "c_kv")
    _check(to_f64(k_pe), rk, bound[:, 512:], "k_pe")


@pytest.mark.parametrize("T,H,D", [(1, 16, 2048), (64, 16, 2048), (33, 128, 1024), (700, 16, 512),
                                   (2108, 16, 2048), (257, 32, 1024)])
def test_o_proj_vs_oracle(T, H, D):
    rng = np.random.default_rng(300 + T + H)
    cfg = L.make_config(H, 64, "bf16")
    a, Wo = _bf16(rng, (T, H, 128)), _bf16(rng, (D, H * 128), (H * 128) ** -0.5)
    y = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg, T, D)
    L.mla_o_proj(cfg, a.to(DEV), Wo.to(DEV), y, ws)
    torch.cuda.synchronize()
    assert L.mla_get_device_status(ws)[0] == 0
    ref = O.o_proj(to_f64(a), to_f64(Wo))
    _check(to_f64(y), ref, _bound(a.reshape(T, -1), Wo, ref), "y")


def test_projections_repeat_bit_for_bit_and_refuse_bad_calls():
    rng = np.random.default_rng(400)
    cfg = L.make_config(16, 64, "bf16")
    x, Wq = _bf16(rng, (3, 2048)).to(DEV), _bf16(rng, (16 * 192, 2048), 2048 ** -0.5).to(DEV)
    q_nope = torch.empty((3, 16, 128), dtype=torch.bfloat16, device=DEV)
    q_pe = torch.empty((3, 16, 64), dtype=torch.bfloat16, device=DEV)
    ws = _ws(cfg, 3, 2048)
    outs = []
    for _ in range(3):
        L.mla_q_proj(cfg, x, Wq, q_nope, q_pe, ws)
        outs.append((q_nope.clone(), q_pe.clone()))
    torch.cuda.synchronize()
    assert all(torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1]) for o in outs)
    with pytest.raises(L.MlaError) as e:
        L.mla_q_proj(cfg, x, Wq, q_nope, q_pe, ws[:128])
    assert e.value.status == 3                                  # workspace too small
    with pytest.raises(L.MlaError) as e:
        L.mla_q_proj(cfg, x[:, :100].contiguous(), Wq[:, :100].contiguous(), q_nope, q_pe, ws)
    assert e.value.status == 2                                  # hidden size not a multiple of 64
    cfg32 = L.make_config(16, 64, "f32")
    with pytest.raises(L.MlaError) as e:
        L.mla_o_proj(cfg32, torch.zeros((3, 16, 128), device=DEV), torch.zeros((64, 2048), device=DEV),
                     torch.zeros((3, 64), device=DEV), ws)
    assert e.value.status == 2                                  # bf16 only


LAYER_CASES = {
    "decode_h16": lambda: W.make("layer_h16", [5, 70, 130, 64], [1] * 4, 16, 64, "bf16", seed=71),
    "prefill_rows_h16": lambda: W.make("layer_pf", [40, 9, 200], [3, 1, 2], 16, 32, "bf16", seed=72),
    "decode_h32_bs16": lambda: W.make("layer_h32", [17, 300], [1, 1], 32, 16, "bf16", seed=73),
}


@pytest.mark.parametrize("name", sorted(LAYER_CASES))
def test_whole_layer_vs_the_naive_oracle(name):
    w = LAYER_CASES[name]()
    s = MlaDecodeStep(w, device=DEV)
    s.layer_setup(2048)
    s.layer_populate()
    y = to_f64(s.layer_step())
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    assert L.mla_get_device_status(s.proj_ws)[0] == 0
    li = s.layer
    ref = np.zeros_like(y)
    for b in range(w.batch):
        tr, qr = w.token_range(b), w.q_range(b)
        ref[qr] = O.mla_layer_naive(li.hidden[tr], w.kv_positions[tr], li.W_q, li.W_kv_a, w.W_uk,
                                    w.W_uv, li.W_o, w.rms_weight, w.rms_eps, w.rope_base,
                                    w.softmax_scale, num_new=qr.stop - qr.start)
    assert_close(y, ref, "bf16", f"layer {name}")
    # kv_a_proj and the cache write on a side stream beside q_proj and the
    # absorption: the same kernels on the same inputs, bit for bit
    first = s.y.clone()
    s.y.fill_(float("nan"))
    side = torch.cuda.Stream()
    s.layer_step(side=side)
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.proj_ws_side)[0] == 0
    assert torch.equal(s.y, first)
