"""mla_decode_paged_noalloc: decode + merge for callers that cannot allocate
device memory, using the library's built-in scratch array.

It must give the same latent output as mla_decode_paged + mla_combine with a
caller-allocated workspace, on two calls in a row (the scratch keeps the
previous call's contents), and must refuse a launch whose workspace does not
fit in the scratch. This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from mla_latent_kv_03_gb300 import libmla as L
from mla_latent_kv_03_gb300 import workloads as W
from mla_latent_kv_03_gb300.step import MlaDecodeStep

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    L.load()


def _noalloc(lib, s, o_lat, status):
    cfg = s.cfg
    return lib.mla_decode_paged_noalloc(
        ctypes.byref(cfg), s.q_abs.data_ptr(), s.cache.data_ptr(), s.cache.shape[0],
        s.block_table.data_ptr(), s.block_table.shape[1], s.seq_lens.data_ptr(),
        s.query_start_loc.data_ptr(), s.seq_lens.shape[0], s.q_abs.shape[0], o_lat.data_ptr(),
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _fitting_ctas(w):
    """The CTA count the no-alloc call runs with when the config leaves it at
    0: the default, or the largest smaller count whose workspace fits."""
    cfg = L.make_config(w.num_heads, w.block_size, w.dtype)
    if L.mla_decode_workspace_size(cfg, w.num_q, w.batch) <= SCRATCH:
        return 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    best = 0
    for c in range(1, sms):
        cfg.num_ctas = c
        if L.mla_decode_workspace_size(cfg, w.num_q, w.batch) <= SCRATCH:
            best = c
    return best


@pytest.mark.parametrize("make", [
    lambda: W.make("na_bf16", [700, 1, 129, 64, 2000], [1, 1, 1, 1, 1], 16, 64, "bf16", seed=51),
    lambda: W.make("na_prefill", [150, 64], [40, 1], 16, 64, "bf16", seed=52),
    lambda: W.tiny(),
])
def test_noalloc_matches_workspace_path_twice(make):
    lib = L.load()
    w = make()
    ctas = _fitting_ctas(w)
    assert ctas != 0 or w.name != "na_prefill"   # prefill tiles need the smaller count
    s = MlaDecodeStep(w, device=DEV, num_ctas=ctas)
    s.populate()
    s.absorb()
    s.decode()                       # mla_decode_paged with a caller workspace
    s.combine()
    torch.cuda.synchronize()
    ref = s.o_lat.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    s.cfg.num_ctas = 0                # the no-alloc call picks the count itself
    for call in range(2):
        o = torch.full_like(s.o_lat, float("nan"))
        assert _noalloc(lib, s, o, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        tol = 1e-6 if w.dtype == "f32" else 1e-5
        np.testing.assert_allclose(o.cpu().numpy(), ref.cpu().numpy(), rtol=0, atol=tol,
                                   err_msg=f"call {call + 1}")


def test_noalloc_refuses_a_workspace_beyond_the_scratch():
    lib = L.load()
    w = W.make("na_big", [64] * 600, [1] * 600, 128, 64, "bf16", seed=53)   # 600 x 8 q-tiles
    s = MlaDecodeStep(w, device=DEV)
    assert L.mla_decode_workspace_size(s.cfg, w.num_q, w.batch) > 16 << 20
    o = torch.zeros_like(s.o_lat)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _noalloc(lib, s, o, status) == 3     # MLA_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0


def test_noalloc_refuses_a_fixed_cta_count_that_does_not_fit():
    """With the caller's own CTA count the call does not shrink it: a count
    whose workspace exceeds the scratch is refused and o_lat is untouched."""
    lib = L.load()
    w = W.make("na_fixed", [300, 65, 1], [1, 1, 1], 16, 64, "bf16", seed=54)
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.absorb()
    s.cfg.num_ctas = 1000          # 1,000 split slots of 32 KB: beyond 16 MiB
    assert L.mla_decode_workspace_size(s.cfg, w.num_q, w.batch) > SCRATCH
    o = torch.full_like(s.o_lat, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _noalloc(lib, s, o, status) == 3
    torch.cuda.synchronize()
    assert bool(torch.all(o == 7.0))
    assert int(status.item()) == 0


def test_noalloc_reports_a_bad_block_through_dev_status():
    """A block-table entry beyond the pool is skipped and its bit
    (MLA_DEV_BAD_BLOCK) reaches the caller's status word; the rows of the other
    sequences still match the workspace path."""
    lib = L.load()
    w = W.make("na_badblk", [130, 200], [1, 1], 16, 64, "bf16", seed=55)
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.absorb()
    s.decode()
    s.combine()
    torch.cuda.synchronize()
    ref = s.o_lat.clone()
    bt = s.block_table.clone()
    s.block_table[0, 1] = s.cache.shape[0] + 5      # sequence 0's second page: out of range
    o = torch.full_like(s.o_lat, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _noalloc(lib, s, o, status) == 0
    torch.cuda.synchronize()
    s.block_table.copy_(bt)
    assert int(status.item()) & 2 == 2                # MLA_DEV_BAD_BLOCK
    q1 = slice(int(w.query_start_loc[1]), int(w.query_start_loc[2]))
    np.testing.assert_allclose(o[q1].cpu().numpy(), ref[q1].cpu().numpy(), rtol=0, atol=1e-5)
    assert bool(torch.isfinite(o).all())
