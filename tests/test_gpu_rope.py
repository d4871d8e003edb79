"""GPU parity of the interleaved RoPE pairing (mla_config.rope_interleaved =
1: pairs (2i, 2i+1) instead of (i, i+32)) at every place the library rotates
a vector -- the cache writes (bf16, fp32, FP8), the query absorption (small,
tensor-core and fp32 paths) and the full K/V form's query -- against the fp64
oracle, through the C ABI."""

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


def _ref_out(w):
    out = np.zeros((w.num_q, w.num_heads, 128))
    for b in range(w.batch):
        tr, qr = w.token_range(b), w.q_range(b)
        if qr.stop == qr.start:
            continue
        out[qr] = O.mla_sequence_naive(
            w.c_kv_raw[tr], w.k_pe_raw[tr], w.kv_positions[tr], w.q_nope[qr], w.q_pe[qr],
            w.q_positions[qr], w.W_uk, w.W_uv, w.rms_weight, w.rms_eps, w.rope_base,
            w.softmax_scale, interleaved=True)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cache_write_rows(dtype):
    w = W.make("ri_cw", [7, 33, 130, 1], [1] * 4, 16, 32, dtype, seed=81)
    s = MlaDecodeStep(w, device=DEV, rope_interleaved=True)
    s.populate()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.status)[0] == 0
    got = to_f64(s.cache).reshape(-1, 576)[w.slot_mapping]
    ref = O.latent_cache_rows(w.c_kv_raw, w.k_pe_raw, w.kv_positions, w.rms_weight, w.rms_eps,
                              w.rope_base, interleaved=True)
    if dtype == "bf16":
        assert np.all(np.abs(got - ref) <= bf16_ulp(ref)), "row values beyond 1 bf16 ulp"
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6)
    # the rotate-half rows differ in the rope part: the flag is honoured
    half = O.latent_cache_rows(w.c_kv_raw, w.k_pe_raw, w.kv_positions, w.rms_weight, w.rms_eps,
                               w.rope_base)
    assert np.max(np.abs(got[:, 512:] - half[:, 512:])) > 0.1


@pytest.mark.parametrize("case", ["small_bf16", "tc_bf16", "f32"])
def test_absorb_rope_part(case):
    if case == "tc_bf16":      # 300 query rows: the tensor-core absorption
        w = W.make("ri_ab_tc", [320, 64], [299, 1], 16, 64, "bf16", seed=82)
    else:
        w = W.make("ri_ab", [40, 9, 200], [3, 1, 2], 32 if case == "small_bf16" else 16, 16,
                   "f32" if case == "f32" else "bf16", seed=83)
    s = MlaDecodeStep(w, device=DEV, rope_interleaved=True)
    s.absorb()
    torch.cuda.synchronize()
    got = to_f64(s.q_abs)
    ref = O.absorb_q(w.q_nope, w.q_pe, w.q_positions, w.W_uk, w.rope_base, interleaved=True)
    tol = bf16_ulp(ref[..., 512:]) if w.dtype == "bf16" else 1e-6
    assert np.all(np.abs(got[..., 512:] - ref[..., 512:]) <= tol)


@pytest.mark.parametrize("name,H,dtype", [("decode", 16, "bf16"), ("prefill", 16, "bf16"),
                                          ("h128", 128, "bf16"), ("fp32", 16, "f32")])
def test_absorbed_step_end_to_end(name, H, dtype):
    if name == "prefill":
        w = W.make("ri_pf", [150, 64, 20], [40, 1, 20], H, 64, dtype, seed=84)
    else:
        w = W.make("ri_" + name, [5, 70, 129, 64], [1] * 4, H, 32, dtype, seed=85)
    s = MlaDecodeStep(w, device=DEV, rope_interleaved=True)
    s.populate()
    out = to_f64(s.step())
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    assert_close(out, _ref_out(w), dtype, f"interleaved {name}")


def test_full_kv_form_end_to_end():
    w = W.make("ri_nv", [33, 97, 300], [1, 1, 1], 16, 64, "bf16", seed=86)
    s = MlaDecodeStep(w, device=DEV, rope_interleaved=True)
    s.naive_setup()
    s.naive_populate()
    s.naive_decode()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.naive_ws)[0] == 0
    assert_close(to_f64(s.out_naive), _ref_out(w), "bf16", "interleaved full K/V")


def test_fp8_cache_rope_part():
    w = W.make("ri_f8", [40, 200], [1, 1], 16, 64, "bf16", seed=87)
    s = MlaDecodeStep(w, device=DEV, rope_interleaved=True)
    s.fp8_setup(0.05)
    s.fp8_populate()
    torch.cuda.synchronize()
    rows = s.cache8.cpu().numpy().reshape(-1, 640)[w.slot_mapping]
    rope = rows[:, 512:].copy().view(np.uint16).astype(np.uint32) << 16
    rope = rope.view(np.float32).astype(np.float64)
    _, k_rot = O.fp8_latent_rows(w.c_kv_raw, w.k_pe_raw, w.kv_positions, w.rms_weight,
                                 w.rms_eps, w.rope_base, 0.05, interleaved=True)
    assert np.all(np.abs(rope - k_rot) <= bf16_ulp(k_rot))


def test_flag_outside_zero_one_is_refused():
    cfg = L.make_config(16, 64, "bf16")
    cfg.rope_interleaved = 2
    q = torch.zeros((1, 16, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(L.MlaError) as e:
        L.mla_absorb_q(cfg, q, torch.zeros((1, 16, 64), dtype=torch.bfloat16, device=DEV),
                       torch.zeros(1, dtype=torch.int32, device=DEV),
                       torch.zeros((16, 512, 128), dtype=torch.bfloat16, device=DEV),
                       torch.zeros((1, 16, 576), dtype=torch.bfloat16, device=DEV))
    assert e.value.status == 1
