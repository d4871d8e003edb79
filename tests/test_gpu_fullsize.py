"""Full-size workloads, in the launch configuration the bench times (one CTA
per SM), checked against the fp64 oracle: the naive form (K and V expanded per
head) on sampled sequences and heads, and the absorbed form (held equal to the
naive one to 1e-12 by the oracle's own tests) on every head of at least 8
sequences per workload, always including the shortest and the longest."""

import numpy as np
import pytest
import torch

from _helpers import assert_close, ref_out, ref_out_absorbed, to_f64
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


# ---------------------------------------------------------------------------
# the step exactly as the bench times it: captured in a CUDA graph (every
# kernel with programmatic dependent launch), replayed, then checked
# ---------------------------------------------------------------------------

def _bench_step(s, w, side, ev_fork, ev_join):
    mixed = bool(w.is_new.sum() > w.batch)
    tc = w.num_heads >= 64 or w.num_q >= 4 * w.batch
    if not tc and w.num_q <= 256:
        s.absorb()
        s.decode_paged_combine()      # plan + decode + split merge, one kernel
        s.out_proj()
        return
    cur = torch.cuda.current_stream()
    ev_fork.record(cur)
    side.wait_event(ev_fork)
    with torch.cuda.stream(side):
        s.plan()
        ev_join.record(side)
    if mixed:
        s.write_new()
    s.absorb()
    cur.wait_event(ev_join)
    s.decode_combine()
    s.out_proj()


def _run_graphed(w, s, steps=3, replays=2):
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
    with torch.cuda.stream(stream):
        _bench_step(s, w, side, ev_fork, ev_join)   # eager once (lazy state)
    stream.synchronize()
    s.out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(steps):
            _bench_step(s, w, side, ev_fork, ev_join)
    with torch.cuda.stream(stream):
        for _ in range(replays):
            g.replay()
    stream.synchronize()


def test_serving_bench_step_graphed_and_the_other_forms():
    w = W.serving()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    s.naive_setup()
    _run_graphed(w, s)
    assert s.device_status()[0][0] == 0
    seqs, heads = [0, 17, 40, 63], list(range(16))
    ref = ref_out(w, seqs=seqs, heads=heads)
    rows = np.concatenate([np.arange(w.q_range(b).start, w.q_range(b).stop) for b in seqs])
    assert_close(to_f64(s.out)[rows], ref[rows], "bf16", "serving, graphed bench step")
    # the pages' other two forms at the same size
    s.naive_populate()
    s.naive_decode()
    torch.cuda.synchronize()
    assert_close(to_f64(s.out_naive)[rows], ref[rows], "bf16", "serving, full K/V cache")
    s.kv_naive.view(torch.int16).fill_(0x7FC1)
    s.latent_expand()
    s.naive_decode()
    torch.cuda.synchronize()
    assert L.mla_get_device_status(s.naive_ws)[0] == 0
    assert_close(to_f64(s.out_naive)[rows], ref[rows], "bf16", "serving, latent re-expanded")


def test_ragged_H128_bench_step_graphed():
    w = W.ragged_h128()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    _run_graphed(w, s)
    assert s.device_status()[0][0] == 0
    lens = w.seq_lens
    seqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 7})
    _check(w, s, seqs, [0, 64, 127], "ragged H=128, graphed bench step")


def test_mixed_bench_step_graphed():
    w = W.mixed()
    s = MlaDecodeStep(w, device=DEV)
    s.populate(include_new=False)
    _run_graphed(w, s)
    (st1, _), (st2, _) = s.device_status()
    assert st1 == 0 and st2 == 0
    _check(w, s, [1, 4, 50], [3, 12], "mixed, graphed bench step")


def _graph_replay(step_fn, steps=3, replays=2):
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step_fn()                      # eager once (lazy state)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(steps):
            step_fn()
    with torch.cuda.stream(stream):
        for _ in range(replays):
            g.replay()
    stream.synchronize()


def test_serving_fp8_bench_step_graphed():
    # bench.py --form fp8: two CTAs per SM, kv_scale 0.02
    w = W.serving()
    s = MlaDecodeStep(w, device=DEV)
    s.fp8_setup(0.02)
    s.fp8_populate()

    def step():
        s.absorb()
        s.decode_paged_combine_fp8()
        s.out_proj()

    s.out.fill_(float("nan"))
    _graph_replay(step)
    assert s.device_status()[0][0] == 0
    seqs = [0, 23, 63]
    q_abs = O.absorb_q(w.q_nope, w.q_pe, w.q_positions, w.W_uk, w.rope_base)
    for b in seqs:
        tr, qr = w.token_range(b), w.q_range(b)
        codes, k_rot = O.fp8_latent_rows(w.c_kv_raw[tr], w.k_pe_raw[tr], w.kv_positions[tr],
                                         w.rms_weight, w.rms_eps, w.rope_base, 0.02)
        rows = np.concatenate([O.e4m3_decode(codes) * 0.02, k_rot], -1)
        o, _ = O.latent_attention(q_abs[qr], rows, w.q_positions[qr], w.softmax_scale)
        assert_close(to_f64(s.out)[qr], O.out_proj(o, w.W_uv), "bf16", f"fp8 serving seq {b}")


def test_serving_layer_bench_step_graphed():
    # bench.py --form layer: hidden states -> q_proj, kv_a_proj + cache write,
    # absorb, decode + merge, out_proj, o_proj (hidden 2048)
    w = W.serving()
    s = MlaDecodeStep(w, device=DEV)
    s.layer_setup(2048)
    s.layer_populate()
    s.y.fill_(float("nan"))
    side = torch.cuda.Stream()
    _graph_replay(lambda: s.layer_step(side=side))   # as the bench runs it
    assert s.device_status()[0][0] == 0
    assert L.mla_get_device_status(s.proj_ws)[0] == 0
    assert L.mla_get_device_status(s.proj_ws_side)[0] == 0
    li = s.layer
    for b in (5, 62):
        tr, qr = w.token_range(b), w.q_range(b)
        ref = O.mla_layer_naive(li.hidden[tr], w.kv_positions[tr], li.W_q, li.W_kv_a, w.W_uk,
                                w.W_uv, li.W_o, w.rms_weight, w.rms_eps, w.rope_base,
                                w.softmax_scale, num_new=1)
        assert_close(to_f64(s.y)[qr], ref, "bf16", f"layer serving seq {b}")


# ---------------------------------------------------------------------------
# every head of many sequences, through the oracle's absorbed form, on the
# step as the bench times it (graphed, fused merges)
# ---------------------------------------------------------------------------

def _check_all_heads(w, s, seqs, what, rows_of=None):
    ref = ref_out_absorbed(w, seqs, rows_of)
    m = ~np.isnan(ref[:, 0, 0])
    assert m.sum() > 0
    return assert_close(to_f64(s.out)[m], ref[m], w.dtype, what)


def test_serving_16_sequences_every_head():
    w = W.serving()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    _run_graphed(w, s)
    assert s.device_status()[0][0] == 0
    seqs = sorted({int(x) for x in np.linspace(0, w.batch - 1, 16)})
    assert len(seqs) == 16
    _check_all_heads(w, s, seqs, "serving, 16 sequences x 16 heads")


def test_ragged_H128_8_sequences_every_head():
    w = W.ragged_h128()
    s = MlaDecodeStep(w, device=DEV)
    s.populate()
    _run_graphed(w, s)
    assert s.device_status()[0][0] == 0
    lens = np.asarray(w.seq_lens)
    order = np.argsort(lens)
    pick = {int(order[0]), int(order[-1])}
    pick |= {int(order[k]) for k in np.linspace(1, len(order) - 2, 6).astype(int)}
    seqs = sorted(pick)
    assert len(seqs) >= 8
    _check_all_heads(w, s, seqs, "ragged H=128, 8 sequences x 128 heads")


def test_mixed_every_prefill_sequence_and_8_decode_sequences_every_head():
    w = W.mixed()
    s = MlaDecodeStep(w, device=DEV)
    s.populate(include_new=False)
    _run_graphed(w, s)
    (st1, _), (st2, _) = s.device_status()
    assert st1 == 0 and st2 == 0
    ql = np.diff(np.asarray(w.query_start_loc))
    prefill = [b for b in range(w.batch) if ql[b] > 1]
    decode = [b for b in range(w.batch) if ql[b] == 1]
    assert len(prefill) == 4
    dec = [decode[int(k)] for k in np.linspace(0, len(decode) - 1, 8).astype(int)]
    # 64 of each prefill chunk's 512 query rows (the first and the last among
    # them), every decode row
    rng = np.random.default_rng(9)

    def rows_of(b):
        n = int(ql[b])
        if n == 1:
            return [0]
        return sorted({0, n - 1} | set(rng.choice(n, 62, replace=False).tolist()))

    _check_all_heads(w, s, prefill + dec, "mixed: 4 prefill + 8 decode sequences x 16 heads",
                     rows_of)


def test_mixed_layer_bench_step_graphed():
    # bench.py --workload mixed --form layer: the projections of the 2,108 new
    # tokens run on the tensor-core projection kernel (from 256 rows)
    w = W.mixed()
    s = MlaDecodeStep(w, device=DEV)
    s.populate(include_new=False)
    s.layer_setup(2048)
    s.layer_populate()
    s.y.fill_(float("nan"))
    side = torch.cuda.Stream()
    _graph_replay(lambda: s.layer_step(side=side))   # as the bench runs it
    assert s.device_status()[0][0] == 0
    assert L.mla_get_device_status(s.proj_ws)[0] == 0
    assert L.mla_get_device_status(s.proj_ws_side)[0] == 0
    li = s.layer
    ql = np.diff(np.asarray(w.query_start_loc))
    got = to_f64(s.y)

    def ref_rows(b):
        tr = w.token_range(b)
        return O.mla_layer_naive(li.hidden[tr], w.kv_positions[tr], li.W_q, li.W_kv_a, w.W_uk,
                                 w.W_uv, li.W_o, w.rms_weight, w.rms_eps, w.rope_base,
                                 w.softmax_scale, num_new=int(ql[b]))

    # a prefill chunk (512 rows), then eight decode sequences (one row each)
    # under one bar, as the other full-size tests sample
    assert_close(got[w.q_range(0)], ref_rows(0), "bf16", "layer mixed, prefill sequence 0")
    dec = [10, 17, 24, 31, 38, 45, 52, 63]
    assert all(ql[b] == 1 for b in dec)
    rows = [w.q_range(b).start for b in dec]
    assert_close(got[rows], np.concatenate([ref_rows(b) for b in dec]), "bf16",
                 "layer mixed, 8 decode sequences")
