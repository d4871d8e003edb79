"""GPU parity of the FP8 latent cache (e4m3 codes of c_hat / kv_scale, then
the bf16 rope key) against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from _helpers import assert_close, bf16_ulp, ref_o_lat_from, to_f64
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


CASES = {
    "ragged_tails_bs64": lambda: W.make("f8_tails", [1, 63, 64, 65, 127, 128, 129, 1000], [1] * 8,
                                        16, 64, "bf16", seed=61, extra_blocks=2),
    "bs16_h32": lambda: W.make("f8_bs16", [5, 40, 200], [1] * 3, 32, 16, "bf16", seed=62),
    "bs32": lambda: W.make("f8_bs32", [33, 97, 2], [1] * 3, 16, 32, "bf16", seed=63),
    "empty_seq": lambda: W.make("f8_empty", [0, 5, 0, 70], [0, 1, 0, 1], 16, 64, "bf16", seed=64),
}


def _step(name, kv_scale, num_ctas=0):
    w = CASES[name]()
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.fp8_setup(kv_scale)
    return w, s


def _dequantised_cache(s):
    """The GPU's own FP8 cache as fp64 rows [num_blocks, bs, 576]."""
    c8 = s.cache8.cpu()
    codes = c8[..., :512].numpy()
    rope = c8[..., 512:].contiguous().view(torch.bfloat16).double().numpy()
    return np.concatenate([O.e4m3_decode(codes) * s.kv_scale, rope], -1)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("kv_scale", [1.0, 0.05])
def test_fp8_cache_write_codes_and_placement(name, kv_scale):
    w, s = _step(name, kv_scale)
    s.cache8.fill_(0x7F)                                    # an e4m3 NaN byte
    s.fp8_populate()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.status)[0] == 0
    rows = s.cache8.cpu().numpy().reshape(-1, 640)
    written = np.zeros(rows.shape[0], dtype=bool)
    written[w.slot_mapping] = True
    assert np.all(rows[~written] == 0x7F), "bytes outside the slots changed"
    got = rows[w.slot_mapping]
    codes_ref, k_rot = O.fp8_latent_rows(w.c_kv_raw, w.k_pe_raw, w.kv_positions, w.rms_weight,
                                         w.rms_eps, w.rope_base, kv_scale)
    # the GPU normalises in fp32: a code may differ only where the exact value
    # lies within fp32 error of a rounding midpoint, and then by one step
    diff = got[:, :512] != codes_ref
    if diff.any():
        x = (O.rms_norm(w.c_kv_raw, w.rms_weight, w.rms_eps) / kv_scale)[diff]
        g, r = O.e4m3_decode(got[:, :512][diff]), O.e4m3_decode(codes_ref[diff])
        mid = (g + r) / 2
        assert np.all(np.abs(x - mid) <= 1e-5 * np.abs(x) + 1e-12), "code off a midpoint"
        assert np.all(np.abs(g - r) <= np.maximum(np.abs(r), 2.0 ** -6) * 2.0 ** -3 + 1e-12)
    assert diff.mean() < 1e-3
    rope = got[:, 512:].copy().view(np.uint16).astype(np.uint32) << 16
    rope = rope.view(np.float32).astype(np.float64)
    assert np.all(np.abs(rope - k_rot) <= bf16_ulp(k_rot)), "rope key beyond 1 bf16 ulp"


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("kv_scale,num_ctas", [(1.0, 0), (0.05, 7), (4.0, 500)])
def test_fp8_decode_vs_oracle_on_the_gpus_cache(name, kv_scale, num_ctas):
    w, s = _step(name, kv_scale, num_ctas)
    s.fp8_populate()
    s.absorb()
    outs = []
    for _ in range(2):
        s.o_lat.fill_(float("nan"))
        s.decode_paged_combine_fp8()
        outs.append(s.o_lat.clone())
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    assert torch.equal(outs[0], outs[1])
    ref = ref_o_lat_from(w, _dequantised_cache(s), to_f64(s.q_abs))
    got = to_f64(outs[0])
    empty = np.isnan(ref).all(axis=(1, 2))
    assert np.all(got[empty] == 0)
    assert_close(got, ref, "bf16", f"fp8 decode {name} scale {kv_scale}")


def test_fp8_end_to_end_against_the_oracles_fp8_path():
    # serving-shaped rows cut into several parts, the oracle quantising from fp64
    w = W.make("f8_srv", [4096] * 8, [1] * 8, 16, 64, "bf16", seed=65)
    s = MlaDecodeStep(w, device=DEV)
    s.fp8_setup(0.02)
    s.fp8_populate()
    s.absorb()
    s.decode_paged_combine_fp8()
    s.out_proj()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    codes, k_rot = O.fp8_latent_rows(w.c_kv_raw, w.k_pe_raw, w.kv_positions, w.rms_weight,
                                     w.rms_eps, w.rope_base, 0.02)
    rows = np.concatenate([O.e4m3_decode(codes) * 0.02, k_rot], -1)
    q_abs = O.absorb_q(w.q_nope, w.q_pe, w.q_positions, w.W_uk, w.rope_base)
    ref = np.zeros((w.num_q, w.num_heads, 128))
    for b in range(w.batch):
        tr, qr = w.token_range(b), w.q_range(b)
        o, _ = O.latent_attention(q_abs[qr], rows[tr], w.q_positions[qr], w.softmax_scale)
        ref[qr] = O.out_proj(o, w.W_uv)
    assert_close(to_f64(s.out), ref, "bf16", "fp8 end to end")


def test_fp8_decode_is_refused_off_its_path():
    w = W.make("f8_h128", [40, 9], [1, 1], 128, 64, "bf16", seed=66)
    s = MlaDecodeStep(w, device=DEV)
    s.fp8_setup(1.0)
    with pytest.raises(L.MlaError) as e:
        s.decode_paged_combine_fp8()
    assert e.value.status == 2
