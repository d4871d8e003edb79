"""The C ABI without a GPU: the library builds and loads, exports every call
that include/mla.h declares, and rejects bad arguments on the host before any
CUDA work (no compute call runs here)."""

import ctypes
import os
import re

import pytest

from mla_latent_kv_03_gb300 import libmla as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return L.load(build_if_missing=True)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mla_cache_write", "mla_absorb_q", "mla_decode_paged", "mla_combine",
                     "mla_out_proj", "mla_decode_workspace_size", "mla_get_device_status"):
        assert required in names
    assert set(names) == set(L.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.mla_version() >= 1


def test_status_strings(lib):
    for code in range(9):
        assert lib.mla_status_string(code)
    assert lib.mla_status_string(0) == b"ok"


def test_default_config_is_v2_lite(lib):
    cfg = L.make_config(16, 64, "bf16")
    assert (cfg.kv_lora_rank, cfg.qk_rope_head_dim, cfg.qk_nope_head_dim, cfg.v_head_dim) == (512, 64, 128, 128)
    assert abs(cfg.softmax_scale - 192 ** -0.5) < 1e-7
    assert cfg.rms_eps == pytest.approx(1e-6) and cfg.rope_base == 10000.0
    assert cfg.dtype == L.MLA_BF16 and cfg.num_ctas == 0


@pytest.mark.parametrize("field,value,expect", [
    ("num_heads", 24, 2), ("num_heads", 256, 2), ("block_size", 128, 2), ("block_size", 8, 2),
    ("kv_lora_rank", 256, 2), ("qk_rope_head_dim", 32, 2), ("dtype", 7, 2), ("num_ctas", -1, 1),
])
def test_unsupported_configs_are_rejected(lib, field, value, expect):
    cfg = L.make_config(16, 64, "bf16")
    setattr(cfg, field, value)
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    s = lib.mla_absorb_q(ctypes.byref(cfg), p, p, p, p, p, 1, None)
    assert s == expect


def test_null_and_misaligned_pointers_are_rejected(lib):
    cfg = L.make_config(16, 64, "bf16")
    p = ctypes.c_void_p(256)
    assert lib.mla_absorb_q(None, p, p, p, p, p, 1, None) == 1
    assert lib.mla_absorb_q(ctypes.byref(cfg), None, p, p, p, p, 1, None) == 1
    assert lib.mla_absorb_q(ctypes.byref(cfg), ctypes.c_void_p(258), p, p, p, p, 1, None) == 1
    assert lib.mla_out_proj(ctypes.byref(cfg), p, p, None, 1, None) == 1
    assert lib.mla_cache_write(ctypes.byref(cfg), p, p, p, ctypes.c_void_p(260), 1, p, p, 4, None, None) == 1
    # zero-sized work is a no-op that succeeds without touching pointers
    assert lib.mla_absorb_q(ctypes.byref(cfg), None, None, None, None, None, 0, None) == 0
    assert lib.mla_cache_write(ctypes.byref(cfg), None, None, None, None, 0, None, None, 0, None, None) == 0


def test_workspace_size_with_fixed_cta_count(lib):
    cfg = L.make_config(16, 64, "bf16", num_ctas=152)
    n64 = lib.mla_decode_workspace_size(ctypes.byref(cfg), 64, 64)
    # 152 CTAs + 64 q-tiles partial slots of 16 x 512 fp32 dominate
    assert n64 >= (152 + 64) * 16 * 512 * 4
    assert n64 < (152 + 64) * 16 * 512 * 4 + 64 * 1024
    cfg128 = L.make_config(128, 64, "bf16", num_ctas=152)
    n128 = lib.mla_decode_workspace_size(ctypes.byref(cfg128), 32, 32)
    assert n128 >= (152 + 32 * 8) * 16 * 512 * 4
    assert lib.mla_decode_workspace_size(None, 1, 1) == 0


def test_decode_rejects_small_workspace_on_host(lib):
    cfg = L.make_config(16, 64, "bf16", num_ctas=8)
    p = ctypes.c_void_p(1 << 20)
    need = lib.mla_decode_workspace_size(ctypes.byref(cfg), 4, 4)
    s = lib.mla_decode_paged(ctypes.byref(cfg), p, p, 16, p, 4, p, p, 4, 4, p, need - 256, None)
    assert s == 3
    s = lib.mla_decode_paged(ctypes.byref(cfg), p, p, 16, p, 4, p, p, 4, 70000, p, 1 << 40, None)
    assert s == 2  # more query rows than one plan holds


def test_naive_forms_are_bf16_only_and_check_their_workspace(lib):
    f32 = L.make_config(16, 64, "f32")
    bf16 = L.make_config(16, 64, "bf16")
    assert lib.mla_naive_workspace_size(ctypes.byref(f32), 4, 4, 4) == 0
    p = ctypes.c_void_p(1 << 20)
    # rejected on the host before any device work
    assert lib.mla_naive_decode(ctypes.byref(f32), p, p, p, p, 16, p, 4, p, p, 4, 4, p,
                                1 << 30, p, None) == 2
    need = lib.mla_naive_workspace_size(ctypes.byref(bf16), 4, 4, 0)
    # the 256-byte header plus the transposed weights [16, 256, 512] bf16, at least
    assert need >= 256 + 16 * 256 * 512 * 2
    assert lib.mla_naive_decode(ctypes.byref(bf16), p, p, p, p, 16, p, 4, p, p, 4, 4, p,
                                256, p, None) == 3
    assert lib.mla_latent_expand(ctypes.byref(bf16), p, 16, p, 4, p, 4, p, p, p, p, 256, None) == 3
    # the two-part expansion: the same refusals, nothing launched
    assert lib.mla_latent_expand_prepare(ctypes.byref(bf16), p, p, p, 256, None) == 3
    assert lib.mla_latent_expand_prepare(ctypes.byref(f32), p, p, p, 1 << 30, None) == 2
    assert lib.mla_latent_expand_prepare(ctypes.byref(bf16), None, p, p, 1 << 30, None) == 1
    assert lib.mla_latent_expand_prepared(ctypes.byref(bf16), p, 16, p, 4, p, 4, p, p, 256, None) == 3
    assert lib.mla_latent_expand_prepared(ctypes.byref(bf16), None, 16, p, 4, p, 4, p, p, 1 << 30,
                                          None) == 1


def test_rope_pairing_field_defaults_to_rotate_half_and_is_checked(lib):
    cfg = L.make_config(16, 64, "bf16")
    assert cfg.rope_interleaved == 0
    assert L.make_config(16, 64, "bf16", rope_interleaved=True).rope_interleaved == 1
    cfg.rope_interleaved = 2
    p = ctypes.c_void_p(256)
    assert lib.mla_absorb_q(ctypes.byref(cfg), p, p, p, p, p, 1, None) == 1


def test_fp8_calls_check_their_arguments_on_the_host(lib):
    bf16 = L.make_config(16, 64, "bf16")
    f32 = L.make_config(16, 64, "f32")
    h128 = L.make_config(128, 64, "bf16")
    p = ctypes.c_void_p(1 << 20)
    f = ctypes.c_float
    assert lib.mla_cache_write_fp8(ctypes.byref(f32), p, p, p, p, 4, p, f(1.0), p, 4, None, None) == 2
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert lib.mla_cache_write_fp8(ctypes.byref(bf16), p, p, p, p, 4, p, f(bad), p, 4, None,
                                       None) == 1
    assert lib.mla_cache_write_fp8(ctypes.byref(bf16), None, None, None, None, 0, None, f(1.0),
                                   None, 0, None, None) == 0
    dec = lib.mla_decode_paged_combine_fp8
    assert dec(ctypes.byref(bf16), p, p, 16, p, 4, p, p, 4, 4, f(0.0), p, 1 << 30, p, None) == 1
    # 128 heads take the tensor-core path, which has no FP8 form
    assert dec(ctypes.byref(h128), p, p, 16, p, 4, p, p, 4, 4, f(1.0), p, 1 << 30, p, None) == 2
    assert lib.mla_decode_fp8_workspace_size(None, 4, 4) == 0


def test_projections_check_their_arguments_on_the_host(lib):
    bf16 = L.make_config(16, 64, "bf16")
    f32 = L.make_config(16, 64, "f32")
    p = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 21)
    assert lib.mla_proj_workspace_size(ctypes.byref(f32), 64, 2048) == 0
    assert lib.mla_proj_workspace_size(ctypes.byref(bf16), 64, 100) == 0
    assert lib.mla_proj_workspace_size(ctypes.byref(bf16), -1, 2048) == 0
    for fn in (lib.mla_q_proj, lib.mla_kv_a_proj):
        assert fn(ctypes.byref(f32), p, p, p, p, 4, 2048, ws, 1 << 20, None) == 2      # bf16 only
        assert fn(ctypes.byref(bf16), p, p, p, p, 4, 2000, ws, 1 << 20, None) == 2     # K % 64
        assert fn(ctypes.byref(bf16), p, p, p, p, 4, 2048, None, 1 << 20, None) == 1   # workspace
        assert fn(ctypes.byref(bf16), p, p, p, p, 4, 2048, ctypes.c_void_p((1 << 21) + 16),
                  1 << 20, None) == 1                                                  # 256-aligned
        assert fn(ctypes.byref(bf16), ctypes.c_void_p((1 << 20) + 2), p, p, p, 4, 2048, ws,
                  1 << 20, None) == 1                                                  # 16-aligned
        assert fn(ctypes.byref(bf16), None, None, None, None, 0, 2048, ws, 256, None) == 0
    assert lib.mla_o_proj(ctypes.byref(bf16), p, p, None, 4, 2048, ws, 1 << 20, None) == 1
    assert lib.mla_o_proj(ctypes.byref(bf16), p, p, p, -1, 2048, ws, 1 << 20, None) == 1


def test_naive_prefill_checks_its_arguments_on_the_host(lib):
    f32 = L.make_config(16, 64, "f32")
    bf16 = L.make_config(16, 64, "bf16")
    p = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 21)
    fn = lib.mla_naive_prefill
    assert fn(ctypes.byref(f32), p, p, p, p, 16, p, 4, p, p, 4, 4, ws, 256, p, None) == 2
    assert fn(ctypes.byref(bf16), p, p, p, p, 16, p, 4, p, p, 4, 4, None, 256, p, None) == 1
    assert fn(ctypes.byref(bf16), p, p, p, p, 16, p, 4, p, p, 4, 4, ws, 128, p, None) == 1
    assert fn(ctypes.byref(bf16), ctypes.c_void_p((1 << 20) + 8), p, p, p, 16, p, 4, p, p, 4, 4,
              ws, 256, p, None) == 1
    assert fn(ctypes.byref(bf16), p, p, p, p, 16, p, 4, p, p, 4, -1, ws, 256, p, None) == 1
    # no rows: nothing to do, nothing touched
    assert fn(ctypes.byref(bf16), None, None, None, None, 16, None, 4, None, None, 4, 0, ws, 256,
              None, None) == 0
    # more query rows than the kernel indexes
    assert fn(ctypes.byref(bf16), p, p, p, p, 16, p, 4, p, p, 4, 1 << 31, ws, 256, p,
              None) == 2


def _decode_args(p, num_q=1, batch=1, num_blocks=4, mbps=4):
    # q_abs, cache, num_blocks, block_table, max_blocks_per_seq, seq_lens,
    # query_start_loc, batch, num_q
    return [p, p, num_blocks, p, mbps, p, p, batch, num_q]


@pytest.mark.parametrize("case", ["cfg", "num_ctas", "batch", "num_q", "blocks", "null_q", "mis_cache",
                                  "mis_seq", "rows"])
def test_noalloc_refuses_like_decode_paged(lib, case):
    """The no-alloc decode runs mla_decode_paged's argument checks before it
    touches its scratch, and returns the same codes."""
    cfg = L.make_config(16, 64, "bf16")
    p = ctypes.c_void_p(256)
    args = _decode_args(p)
    cfgp = ctypes.byref(cfg)
    if case == "cfg":
        cfg.num_heads = 24
    elif case == "num_ctas":
        cfg.num_ctas = -2
    elif case == "batch":
        args[7] = -1
    elif case == "num_q":
        args[8] = -1
    elif case == "blocks":
        args[2] = -1
    elif case == "null_q":
        args[0] = None
    elif case == "mis_cache":
        args[1] = ctypes.c_void_p(264)
    elif case == "mis_seq":
        args[5] = ctypes.c_void_p(258)
    elif case == "rows":
        args[8] = 48 * 1024 + 1
    ws = ctypes.c_void_p(4096)
    want = lib.mla_decode_paged(cfgp, *args, ws, 1 << 30, None)
    assert want != 0
    got = lib.mla_decode_paged_noalloc(cfgp, *args, p, None, None)
    assert got == want, (case, got, want)


def test_noalloc_with_no_rows_is_a_noop(lib):
    cfg = L.make_config(16, 64, "bf16")
    assert lib.mla_decode_paged_noalloc(ctypes.byref(cfg), None, None, 0, None, 0, None, None, 0, 0,
                                        None, None, None) == 0


def test_workspace_init_checks_its_arguments(lib):
    ws = ctypes.c_void_p(1 << 20)   # never dereferenced: every case below is refused first
    assert lib.mla_workspace_init(None, 4096, None) == 1
    assert lib.mla_workspace_init(ctypes.c_void_p((1 << 20) + 16), 4096, None) == 1   # not 256-aligned
    assert lib.mla_workspace_init(ws, 8, None) == 1                                   # smaller than the header


def test_plan_checks_its_arguments_on_the_host(lib):
    cfg = L.make_config(16, 64, "bf16")
    c = ctypes.byref(cfg)
    ws, p = ctypes.c_void_p(1 << 20), ctypes.c_void_p(4096)
    assert lib.mla_decode_plan(None, p, p, 1, 1, 4, ws, 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, p, p, 1, -1, 4, ws, 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, p, p, -1, 1, 4, ws, 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, p, p, 1, 1, -4, ws, 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, p, p, 1, 48 * 1024 + 1, 4, ws, 1 << 30, None) == 2   # rows beyond one plan
    assert lib.mla_decode_plan(c, p, p, 1, 1, 4, None, 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, p, p, 1, 1, 4, ctypes.c_void_p((1 << 20) + 64), 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, None, p, 1, 1, 4, ws, 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, p, None, 1, 1, 4, ws, 1 << 30, None) == 1
    assert lib.mla_decode_plan(c, p, p, 0, 1, 4, ws, 1 << 30, None) == 1               # rows without sequences
    assert lib.mla_decode_plan(c, ctypes.c_void_p(4098), p, 1, 1, 4, ws, 1 << 30, None) == 1
    # no rows: nothing to plan, nothing read
    assert lib.mla_decode_plan(c, None, None, 0, 0, 0, ws, 0, None) == 0


@pytest.mark.parametrize("call", ["mla_decode_planned", "mla_decode_combine"])
def test_planned_decode_checks_its_arguments_on_the_host(lib, call):
    cfg = L.make_config(16, 64, "bf16")
    c = ctypes.byref(cfg)
    ws, p, o = ctypes.c_void_p(1 << 20), ctypes.c_void_p(4096), ctypes.c_void_p(8192)
    fn = getattr(lib, call)
    extra = [o] if call == "mla_decode_combine" else []

    def run(cfgp, q, cache, nblk, bt, mbps, batch, nq, w):
        return fn(cfgp, q, cache, nblk, bt, mbps, batch, nq, w, 1 << 30, *extra, None)

    assert run(None, p, p, 8, p, 4, 1, 1, ws) == 1
    assert run(c, p, p, -1, p, 4, 1, 1, ws) == 1
    assert run(c, p, p, 8, p, -4, 1, 1, ws) == 1
    assert run(c, p, p, 8, p, 4, -1, 1, ws) == 1
    assert run(c, p, p, 8, p, 4, 1, -1, ws) == 1
    assert run(c, p, p, 8, p, 4, 1, 48 * 1024 + 1, ws) == 2
    assert run(c, p, p, (1 << 31) // 64 + 1, p, 4, 1, 1, ws) == 2        # slots beyond 2^31
    assert run(c, p, p, 8, p, 4, 1, 1, None) == 1
    assert run(c, None, p, 8, p, 4, 1, 1, ws) == 1
    assert run(c, p, None, 8, p, 4, 1, 1, ws) == 1
    assert run(c, p, p, 8, None, 4, 1, 1, ws) == 1
    assert run(c, ctypes.c_void_p(4104), p, 8, p, 4, 1, 1, ws) == 1      # q_abs not 16-byte aligned
    assert run(c, p, p, 8, ctypes.c_void_p(4098), 4, 1, 1, ws) == 1      # block table not 4-byte aligned
    assert run(c, None, None, 0, None, 0, 0, 0, ws) == 0                  # no rows
    if call == "mla_decode_combine":
        assert fn(c, p, p, 8, p, 4, 1, 1, ws, 1 << 30, None, None) == 1                  # no o_lat
        assert fn(c, p, p, 8, p, 4, 1, 1, ws, 1 << 30, ctypes.c_void_p(8200), None) == 1  # o_lat misaligned


def test_combine_calls_check_their_arguments_on_the_host(lib):
    cfg = L.make_config(16, 64, "bf16")
    c = ctypes.byref(cfg)
    ws, o, w = ctypes.c_void_p(1 << 20), ctypes.c_void_p(8192), ctypes.c_void_p(16384)
    assert lib.mla_combine(None, ws, 1 << 30, 1, 1, o, None) == 1
    assert lib.mla_combine(c, ws, 1 << 30, -1, 1, o, None) == 1
    assert lib.mla_combine(c, ws, 1 << 30, 1, -1, o, None) == 1
    assert lib.mla_combine(c, ws, 1 << 30, 1, 48 * 1024 + 1, o, None) == 2
    assert lib.mla_combine(c, None, 1 << 30, 1, 1, o, None) == 1
    assert lib.mla_combine(c, ws, 1 << 30, 1, 1, None, None) == 1
    assert lib.mla_combine(c, ws, 1 << 30, 1, 1, ctypes.c_void_p(8196), None) == 1
    assert lib.mla_combine(c, None, 0, 0, 0, None, None) == 0
    assert lib.mla_combine_out_proj(None, ws, 1 << 30, 1, 1, w, o, None) == 1
    assert lib.mla_combine_out_proj(c, ws, 1 << 30, 1, -1, w, o, None) == 1
    assert lib.mla_combine_out_proj(c, ws, 1 << 30, 1, 48 * 1024 + 1, w, o, None) == 2
    assert lib.mla_combine_out_proj(c, None, 1 << 30, 1, 1, w, o, None) == 1
    assert lib.mla_combine_out_proj(c, ws, 1 << 30, 1, 1, None, o, None) == 1
    assert lib.mla_combine_out_proj(c, ws, 1 << 30, 1, 1, w, None, None) == 1
    assert lib.mla_combine_out_proj(c, ws, 1 << 30, 1, 1, ctypes.c_void_p(16392), o, None) == 1
    assert lib.mla_combine_out_proj(c, None, 0, 0, 0, None, None, None) == 0


def test_naive_cache_write_checks_its_arguments_on_the_host(lib):
    cfg = L.make_config(16, 64, "bf16")
    c = ctypes.byref(cfg)
    ws, p, s8 = ctypes.c_void_p(1 << 20), ctypes.c_void_p(4096), ctypes.c_void_p(8192)

    def run(cfgp, ckv, kpe, pos, slots, n, rms, wuk, wuv, kv, nblk, w, wsb):
        return lib.mla_naive_cache_write(cfgp, ckv, kpe, pos, slots, n, rms, wuk, wuv, kv, nblk, w, wsb, None)

    assert run(None, p, p, p, s8, 4, p, p, p, p, 8, ws, 1 << 30) == 1
    assert run(c, p, p, p, s8, -1, p, p, p, p, 8, ws, 1 << 30) == 1
    assert run(c, p, p, p, s8, 4, p, p, p, p, -8, ws, 1 << 30) == 1
    assert run(c, p, p, p, s8, (1 << 24) + 1, p, p, p, p, 8, ws, 1 << 30) == 1
    assert run(c, p, p, p, s8, 4, p, p, p, p, 8, None, 1 << 30) == 1
    assert run(c, None, p, p, s8, 4, p, p, p, p, 8, ws, 1 << 30) == 1
    assert run(c, p, p, p, s8, 4, p, None, p, p, 8, ws, 1 << 30) == 1
    assert run(c, p, p, p, s8, 4, p, p, p, None, 8, ws, 1 << 30) == 1
    assert run(c, p, p, p, ctypes.c_void_p(8196), 4, p, p, p, p, 8, ws, 1 << 30) == 1   # slots not 8-byte aligned
    assert run(c, p, p, p, s8, 4, p, ctypes.c_void_p(4100), p, p, 8, ws, 1 << 30) == 1  # W_uk misaligned
    assert run(c, p, p, p, s8, 4, p, p, p, p, 8, ws, 64) == 3                          # workspace too small
    assert run(c, None, None, None, None, 0, None, None, None, None, 0, ws, 0) == 0      # no tokens
    f32 = L.make_config(16, 64, "f32")
    assert run(ctypes.byref(f32), p, p, p, s8, 4, p, p, p, p, 8, ws, 1 << 30) == 2      # bf16 only


def test_paged_combine_checks_its_arguments_on_the_host(lib):
    cfg = L.make_config(16, 64, "bf16")
    c = ctypes.byref(cfg)
    ws, p, o = ctypes.c_void_p(1 << 20), ctypes.c_void_p(4096), ctypes.c_void_p(8192)

    def run(cfgp, q, cache, nblk, bt, mbps, sl, qsl, batch, nq, w, out):
        return lib.mla_decode_paged_combine(cfgp, q, cache, nblk, bt, mbps, sl, qsl, batch, nq, w,
                                            1 << 30, out, None)

    assert run(None, p, p, 8, p, 4, p, p, 1, 1, ws, o) == 1
    assert run(c, p, p, 8, p, 4, p, p, 1, -1, ws, o) == 1
    assert run(c, p, p, 8, p, 4, p, p, 1, 48 * 1024 + 1, ws, o) == 2
    assert run(c, p, p, (1 << 31) // 64 + 1, p, 4, p, p, 1, 1, ws, o) == 2
    assert run(c, p, p, 8, p, 4, p, p, 1, 1, None, o) == 1
    assert run(c, p, p, 8, p, 4, None, p, 1, 1, ws, o) == 1          # no seq_lens
    assert run(c, p, p, 8, p, 4, p, None, 1, 1, ws, o) == 1          # no query_start_loc
    assert run(c, p, p, 8, p, 4, p, p, 0, 1, ws, o) == 1             # rows without sequences
    assert run(c, p, p, 8, p, 4, p, p, 1, 1, ws, None) == 1          # no o_lat
    assert run(c, p, p, 8, p, 4, p, p, 1, 1, ws, ctypes.c_void_p(8200)) == 1
    assert run(c, p, p, 8, p, 4, ctypes.c_void_p(4098), p, 1, 1, ws, o) == 1
    assert run(c, None, None, 0, None, 0, None, None, 0, 0, ws, None) == 0


def test_device_status_and_self_test_check_their_arguments(lib):
    word = ctypes.c_uint32(0)
    assert lib.mla_get_device_status(None, ctypes.byref(word), 0, None) == 1
    assert lib.mla_get_device_status(ctypes.c_void_p(4098), ctypes.byref(word), 0, None) == 1
    p = ctypes.c_void_p(4096)
    assert lib.mla_selftest_wait_timeout(None, 1000, None) == 1
    assert lib.mla_selftest_wait_timeout(p, 0, None) == 1
    assert lib.mla_selftest_wait_timeout(p, 10_000_000_001, None) == 1   # limit above 10 s
