"""Full-size workloads, in the launch configuration the bench times (one CTA
per SM), checked against the naive fp64 oracle on sampled sequences and
heads (the oracle expands K and V per head, so every row of every head would
take minutes)."""

import numpy as np
import pytest
import torch

from _helpers import assert_close, ref_out, to_f64
from mla_latent_kv_03_gb300 import libmla as L
from mla_latent_kv_03_gb300 import workloads as W
from mla_latent_kv_03_gb300.step import MlaDecodeStep

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    L.load()


def _check(w, s, seqs, heads, what):
    got = to_f64(s.out)[:, heads]
    ref = ref_out(w, seqs=seqs, heads=heads)
    rows = np.concatenate([np.arange(w.q_range(b).start, w.q_range(b).stop) for b in seqs])
    return assert_close(got[rows], ref[rows], w.dtype, what)


def test_serving_B64_L4096_sampled():
    w = W.serving()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.step()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    _check(w, s, [0, 17, 40, 63], list(range(16)), "serving B=64 L=4096")


def test_ragged_H128_sampled():
    w = W.ragged_h128()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.step()
    torch.cuda.synchronize()
    assert s.device_status()[0][0] == 0
    lens = w.seq_lens
    seqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 3, 20})
    _check(w, s, seqs, [0, 1, 63, 64, 127], "ragged H=128")


def test_mixed_prefill_decode_sampled():
    w = W.mixed()
    s = MlaDecodeStep(w, device=DEV)
    s.populate(include_new=False)     # history only
    s.step(write_new=True)            # this step writes its own new tokens
    torch.cuda.synchronize()
    (st1, _), (st2, _) = s.device_status()
    assert st1 == 0 and st2 == 0
    _check(w, s, [0, 3, 4, 63], [0, 5, 15], "mixed prefill + decode")
