"""Stress of the split merges that run inside the decode kernels.

The CTA that finishes a q-tile's (or q-block half's) last part merges every
part while the others may have finished microseconds earlier on other SMs; the
parts are published with per-thread fences, a CTA barrier and an
acquire-release count (the publish protocol of the kernels' common header).
A visibility flaw there shows up as a rare wrong part in the merge, so these
tests run the fused paths with many parts per row for 200 launches each and
require every launch to equal the first bit for bit (the merge order is fixed,
whichever CTA merges) and the first to meet the parity bars against the
latent-attention oracle on the GPU's own cache rows and absorbed queries.
"""

import numpy as np
import pytest
import torch

from mla_latent_kv_03_gb300 import libmla as L
from mla_latent_kv_03_gb300 import workloads as W
from mla_latent_kv_03_gb300.step import MlaDecodeStep

from _helpers import assert_close, ref_o_lat_from, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LAUNCHES = 200


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    L.load()


def _repeat(s, call, n=LAUNCHES):
    s.o_lat.fill_(float("nan"))
    call()
    first = s.o_lat.clone()
    bad = []
    for i in range(1, n):
        s.o_lat.fill_(float("nan"))
        call()
        if not torch.equal(s.o_lat, first):
            bad.append(i)
    torch.cuda.synchronize()
    assert not bad, f"launches {bad[:10]} differ from the first"
    assert s.device_status()[0][0] == 0
    return first


def _parts_of_longest(w, num_ctas, qtile_units):
    """Parts the longest row is cut into: its tiles over the share size."""
    tiles = [(int(L_) + 63) // 64 for L_ in w.seq_lens]
    units = sum(t * qtile_units for t in tiles)
    share = -(-units // num_ctas)
    return -(-max(tiles) // share)


def test_16_head_self_planned_merge_with_256_parts():
    # 150 q-tiles over 500 CTAs keeps the merge in the kernel; the
    # 32,768-token row (512 tiles, 2 per CTA) is cut into 256 parts
    lens = [32768] + [64] * 149
    w = W.make("stress16", lens, [1] * len(lens), 16, 64, "bf16", seed=71)
    assert _parts_of_longest(w, 500, 1) >= 24
    s = MlaDecodeStep(w, device=DEV, num_ctas=500)
    s.populate()
    s.absorb()
    first = _repeat(s, s.decode_paged_combine)
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(to_f64(first), ref, "bf16", "self-planned fused merge, 256 parts")


def test_16_head_planned_merge_with_many_parts():
    lens = [20000, 9000] + [64] * 148
    w = W.make("stress16p", lens, [1] * len(lens), 16, 64, "bf16", seed=72)
    assert _parts_of_longest(w, 500, 1) >= 24
    s = MlaDecodeStep(w, device=DEV, num_ctas=500)
    s.populate()
    s.absorb()
    s.plan()
    first = _repeat(s, s.decode_combine)
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(to_f64(first), ref, "bf16", "planned fused merge")


@pytest.mark.parametrize("lens,num_ctas", [
    ([32768, 32768] + [64] * 80, 0),      # > 16 parts per half: the row-per-thread merge
    ([8192] + [64] * 30, 40),             # <= 16 parts: the staged-weight merge
])
def test_tensor_core_merge_with_many_parts(lens, num_ctas):
    w = W.make("stress128", lens, [1] * len(lens), 128, 64, "bf16", seed=73)
    s = MlaDecodeStep(w, device=DEV, num_ctas=num_ctas)
    s.populate()
    s.absorb()
    s.plan()
    first = _repeat(s, s.decode_combine)
    ref = ref_o_lat_from(w, to_f64(s.cache), to_f64(s.q_abs))
    assert_close(to_f64(first), ref, "bf16", "tensor-core fused merge")
    s.decode_planned()                                   # partials + the merge kernel
    s.combine()
    np.testing.assert_allclose(to_f64(s.o_lat), to_f64(first), rtol=0, atol=1e-5)
