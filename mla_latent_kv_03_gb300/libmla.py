"""Thin ctypes binding over libmla.so (argument marshalling only).

The functions carry the C names of include/mla.h and take torch tensors for
device buffers; each one checks dtype, device and contiguity, passes raw
pointers and the current CUDA stream to the library, and raises MlaError on a
non-OK status. No computation happens here, and there is no fallback: if
libmla.so cannot be loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

MLA_OK = 0
MLA_F32, MLA_BF16 = 0, 1
STATUS_NAMES = {
    0: "MLA_OK", 1: "MLA_ERR_INVALID_ARGUMENT", 2: "MLA_ERR_UNSUPPORTED",
    3: "MLA_ERR_WORKSPACE_TOO_SMALL", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT",
    6: "MLA_ERR_BAD_BLOCK", 7: "MLA_ERR_BAD_SEQ", 8: "MLA_ERR_BAD_SLOT",
}
DEV_TIMEOUT, DEV_BAD_BLOCK, DEV_BAD_SEQ, DEV_BAD_SLOT = 1, 2, 4, 8

EXPORTS = (
    "mla_default_config", "mla_cache_write", "mla_absorb_q", "mla_decode_workspace_size",
    "mla_workspace_init", "mla_decode_paged", "mla_decode_plan", "mla_decode_planned",
    "mla_decode_combine", "mla_decode_paged_combine", "mla_decode_paged_noalloc",
    "mla_combine_out_proj", "mla_cache_write_fp8", "mla_decode_fp8_workspace_size",
    "mla_decode_paged_combine_fp8",
    "mla_proj_workspace_size", "mla_q_proj", "mla_kv_a_proj", "mla_o_proj",
    "mla_naive_workspace_size", "mla_naive_cache_write",
    "mla_latent_expand", "mla_latent_expand_prepare", "mla_latent_expand_prepared",
    "mla_naive_decode", "mla_naive_prefill",
    "mla_combine", "mla_out_proj",
    "mla_get_device_status", "mla_selftest_wait_timeout", "mla_status_string", "mla_version",
)


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({_status_string(status)})")


class MlaConfig(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32), ("kv_lora_rank", ctypes.c_int32),
        ("qk_rope_head_dim", ctypes.c_int32), ("qk_nope_head_dim", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float), ("rms_eps", ctypes.c_float),
        ("rope_base", ctypes.c_float), ("dtype", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
        ("rope_interleaved", ctypes.c_int32),
    ]


_LIB: Optional[ctypes.CDLL] = None

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_cfgp = ctypes.POINTER(MlaConfig)
_SIGS = {
    "mla_default_config": (None, [_cfgp, _i32, _i32, _i32]),
    "mla_cache_write": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp]),
    "mla_absorb_q": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _vp, _i64, _vp]),
    "mla_decode_workspace_size": (_sz, [_cfgp, _i64, _i32]),
    "mla_decode_fp8_workspace_size": (_sz, [_cfgp, _i64, _i32]),
    "mla_proj_workspace_size": (_sz, [_cfgp, _i64, _i32]),
    "mla_q_proj": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _i64, _i32, _vp, _sz, _vp]),
    "mla_kv_a_proj": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _i64, _i32, _vp, _sz, _vp]),
    "mla_o_proj": (_i32, [_cfgp, _vp, _vp, _vp, _i64, _i32, _vp, _sz, _vp]),
    "mla_workspace_init": (_i32, [_vp, _sz, _vp]),
    "mla_decode_paged": (_i32, [_cfgp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i64, _vp, _sz, _vp]),
    "mla_decode_plan": (_i32, [_cfgp, _vp, _vp, _i32, _i64, _i32, _vp, _sz, _vp]),
    "mla_decode_planned": (_i32, [_cfgp, _vp, _vp, _i64, _vp, _i32, _i32, _i64, _vp, _sz, _vp]),
    "mla_decode_combine": (_i32, [_cfgp, _vp, _vp, _i64, _vp, _i32, _i32, _i64, _vp, _sz, _vp, _vp]),
    "mla_decode_paged_combine": (_i32, [_cfgp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i64,
                                        _vp, _sz, _vp, _vp]),
    "mla_decode_paged_noalloc": (_i32, [_cfgp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i64,
                                        _vp, _vp, _vp]),
    "mla_cache_write_fp8": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _i64, _vp, ctypes.c_float, _vp,
                                   _i64, _vp, _vp]),
    "mla_decode_paged_combine_fp8": (_i32, [_cfgp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32,
                                            _i64, ctypes.c_float, _vp, _sz, _vp, _vp]),
    "mla_naive_workspace_size": (_sz, [_cfgp, _i64, _i32, _i64]),
    "mla_naive_cache_write": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _i64,
                                     _vp, _sz, _vp]),
    "mla_latent_expand_prepare": (_i32, [_cfgp, _vp, _vp, _vp, _sz, _vp]),
    "mla_latent_expand_prepared": (_i32, [_cfgp, _vp, _i64, _vp, _i32, _vp, _i32, _vp, _vp, _sz,
                                          _vp]),
    "mla_latent_expand": (_i32, [_cfgp, _vp, _i64, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _sz,
                                 _vp]),
    "mla_naive_decode": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i64,
                                _vp, _sz, _vp, _vp]),
    "mla_naive_prefill": (_i32, [_cfgp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i64,
                                 _vp, _sz, _vp, _vp]),
    "mla_combine": (_i32, [_cfgp, _vp, _sz, _i32, _i64, _vp, _vp]),
    "mla_combine_out_proj": (_i32, [_cfgp, _vp, _sz, _i32, _i64, _vp, _vp, _vp]),
    "mla_out_proj": (_i32, [_cfgp, _vp, _vp, _vp, _i64, _vp]),
    "mla_get_device_status": (_i32, [_vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, _vp]),
    "mla_selftest_wait_timeout": (_i32, [_vp, _i64, _vp]),
    "mla_status_string": (ctypes.c_char_p, [_i32]),
    "mla_version": (_i32, []),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmla.so (building it first if it is missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libmla.so not found at {path}; run build() first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _status_string(s: int) -> str:
    try:
        return load().mla_status_string(s).decode()
    except Exception:  # the library itself failed to load
        return "?"


def _check(status: int, where: str) -> None:
    if status != MLA_OK:
        raise MlaError(status, where)


def make_config(num_heads: int, block_size: int, dtype: str, num_ctas: int = 0,
                softmax_scale: Optional[float] = None, rms_eps: Optional[float] = None,
                rope_base: Optional[float] = None, rope_interleaved: bool = False) -> MlaConfig:
    cfg = MlaConfig()
    load().mla_default_config(ctypes.byref(cfg), num_heads, block_size,
                              MLA_BF16 if dtype == "bf16" else MLA_F32)
    cfg.num_ctas = num_ctas
    if softmax_scale is not None:
        cfg.softmax_scale = softmax_scale
    if rms_eps is not None:
        cfg.rms_eps = rms_eps
    if rope_base is not None:
        cfg.rope_base = rope_base
    cfg.rope_interleaved = int(bool(rope_interleaved))
    return cfg


def _torch_dtype(cfg: MlaConfig):
    return torch.bfloat16 if cfg.dtype == MLA_BF16 else torch.float32


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def mla_cache_write(cfg: MlaConfig, c_kv, k_pe, positions, slot_mapping, rms_weight, cache,
                    dev_status=None, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_cache_write(
        ctypes.byref(cfg), _ptr(c_kv, dt, "c_kv"), _ptr(k_pe, dt, "k_pe"),
        _ptr(positions, torch.int32, "positions"), _ptr(slot_mapping, torch.int64, "slot_mapping"),
        c_kv.shape[0], _ptr(rms_weight, dt, "rms_weight"), _ptr(cache, dt, "cache"),
        cache.shape[0], _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)),
        "mla_cache_write")


def mla_absorb_q(cfg: MlaConfig, q_nope, q_pe, q_positions, W_uk, q_abs, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_absorb_q(
        ctypes.byref(cfg), _ptr(q_nope, dt, "q_nope"), _ptr(q_pe, dt, "q_pe"),
        _ptr(q_positions, torch.int32, "q_positions"), _ptr(W_uk, dt, "W_uk"),
        _ptr(q_abs, dt, "q_abs"), q_nope.shape[0], _stream(stream)), "mla_absorb_q")


def mla_decode_workspace_size(cfg: MlaConfig, num_q: int, batch: int) -> int:
    return int(load().mla_decode_workspace_size(ctypes.byref(cfg), num_q, batch))


def mla_decode_fp8_workspace_size(cfg: MlaConfig, num_q: int, batch: int) -> int:
    return int(load().mla_decode_fp8_workspace_size(ctypes.byref(cfg), num_q, batch))


def mla_workspace_init(workspace, stream=None) -> None:
    _check(load().mla_workspace_init(_ptr(workspace, None, "workspace"), workspace.numel() *
                                     workspace.element_size(), _stream(stream)),
           "mla_workspace_init")


def mla_decode_paged(cfg: MlaConfig, q_abs, cache, block_table, seq_lens, query_start_loc,
                     workspace, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_decode_paged(
        ctypes.byref(cfg), _ptr(q_abs, dt, "q_abs"), _ptr(cache, dt, "cache"), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(query_start_loc, torch.int32, "query_start_loc"),
        seq_lens.shape[0], q_abs.shape[0], _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)), "mla_decode_paged")


def mla_decode_paged_combine(cfg: MlaConfig, q_abs, cache, block_table, seq_lens,
                             query_start_loc, workspace, o_lat, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_decode_paged_combine(
        ctypes.byref(cfg), _ptr(q_abs, dt, "q_abs"), _ptr(cache, dt, "cache"), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(query_start_loc, torch.int32, "query_start_loc"),
        seq_lens.shape[0], q_abs.shape[0], _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(o_lat, torch.float32, "o_lat"),
        _stream(stream)), "mla_decode_paged_combine")


def mla_decode_plan(cfg: MlaConfig, seq_lens, query_start_loc, num_q: int,
                    max_blocks_per_seq: int, workspace, stream=None) -> None:
    _check(load().mla_decode_plan(
        ctypes.byref(cfg), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(query_start_loc, torch.int32, "query_start_loc"), seq_lens.shape[0], num_q,
        max_blocks_per_seq, _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)), "mla_decode_plan")


def mla_decode_planned(cfg: MlaConfig, q_abs, cache, block_table, batch: int, workspace,
                       stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_decode_planned(
        ctypes.byref(cfg), _ptr(q_abs, dt, "q_abs"), _ptr(cache, dt, "cache"), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1], batch, q_abs.shape[0],
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "mla_decode_planned")


def mla_decode_combine(cfg: MlaConfig, q_abs, cache, block_table, batch: int, workspace, o_lat,
                       stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_decode_combine(
        ctypes.byref(cfg), _ptr(q_abs, dt, "q_abs"), _ptr(cache, dt, "cache"), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1], batch, q_abs.shape[0],
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(o_lat, torch.float32, "o_lat"), _stream(stream)), "mla_decode_combine")


def mla_decode_paged_noalloc(cfg: MlaConfig, q_abs, cache, block_table, seq_lens,
                             query_start_loc, o_lat, dev_status=None, stream=None) -> None:
    """Decode + merge with the library's built-in scratch instead of a workspace."""
    dt = _torch_dtype(cfg)
    _check(load().mla_decode_paged_noalloc(
        ctypes.byref(cfg), _ptr(q_abs, dt, "q_abs"), _ptr(cache, dt, "cache"), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(query_start_loc, torch.int32, "query_start_loc"),
        seq_lens.shape[0], q_abs.shape[0], _ptr(o_lat, torch.float32, "o_lat"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)), "mla_decode_paged_noalloc")


def mla_cache_write_fp8(cfg: MlaConfig, c_kv, k_pe, positions, slot_mapping, rms_weight,
                        kv_scale: float, cache8, status, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_cache_write_fp8(
        ctypes.byref(cfg), _ptr(c_kv, dt, "c_kv"), _ptr(k_pe, dt, "k_pe"),
        _ptr(positions, torch.int32, "positions"), _ptr(slot_mapping, torch.int64, "slot_mapping"),
        c_kv.shape[0], _ptr(rms_weight, dt, "rms_weight"), float(kv_scale),
        _ptr(cache8, torch.uint8, "cache8"), cache8.shape[0], _ptr(status, None, "status"),
        _stream(stream)), "mla_cache_write_fp8")


def mla_decode_paged_combine_fp8(cfg: MlaConfig, q_abs, cache8, block_table, seq_lens,
                                 query_start_loc, kv_scale: float, workspace, o_lat,
                                 stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_decode_paged_combine_fp8(
        ctypes.byref(cfg), _ptr(q_abs, dt, "q_abs"), _ptr(cache8, torch.uint8, "cache8"),
        cache8.shape[0], _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(query_start_loc, torch.int32, "query_start_loc"),
        seq_lens.shape[0], q_abs.shape[0], float(kv_scale), _ptr(workspace, None, "workspace"),
        _nbytes(workspace), _ptr(o_lat, torch.float32, "o_lat"), _stream(stream)),
        "mla_decode_paged_combine_fp8")


def mla_naive_workspace_size(cfg: MlaConfig, num_q: int, max_blocks_per_seq: int,
                             num_tokens: int) -> int:
    return int(load().mla_naive_workspace_size(ctypes.byref(cfg), num_q, max_blocks_per_seq,
                                               num_tokens))


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def mla_naive_cache_write(cfg: MlaConfig, c_kv, k_pe, positions, slot_mapping, rms_weight, W_uk,
                          W_uv, kv_cache, workspace, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_naive_cache_write(
        ctypes.byref(cfg), _ptr(c_kv, dt, "c_kv"), _ptr(k_pe, dt, "k_pe"),
        _ptr(positions, torch.int32, "positions"), _ptr(slot_mapping, torch.int64, "slot_mapping"),
        c_kv.shape[0], _ptr(rms_weight, dt, "rms_weight"), _ptr(W_uk, dt, "W_uk"),
        _ptr(W_uv, dt, "W_uv"), _ptr(kv_cache, dt, "kv_cache"), kv_cache.shape[0],
        _ptr(workspace, None, "workspace"), _nbytes(workspace), _stream(stream)),
        "mla_naive_cache_write")


def mla_latent_expand(cfg: MlaConfig, cache, block_table, seq_lens, W_uk, W_uv, kv_cache,
                      workspace, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_latent_expand(
        ctypes.byref(cfg), _ptr(cache, dt, "cache"), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0], _ptr(W_uk, dt, "W_uk"),
        _ptr(W_uv, dt, "W_uv"), _ptr(kv_cache, dt, "kv_cache"),
        _ptr(workspace, None, "workspace"), _nbytes(workspace), _stream(stream)),
        "mla_latent_expand")


def mla_latent_expand_prepare(cfg: MlaConfig, W_uk, W_uv, workspace, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_latent_expand_prepare(
        ctypes.byref(cfg), _ptr(W_uk, dt, "W_uk"), _ptr(W_uv, dt, "W_uv"),
        _ptr(workspace, None, "workspace"), _nbytes(workspace), _stream(stream)),
        "mla_latent_expand_prepare")


def mla_latent_expand_prepared(cfg: MlaConfig, cache, block_table, seq_lens, kv_cache, workspace,
                               stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_latent_expand_prepared(
        ctypes.byref(cfg), _ptr(cache, dt, "cache"), cache.shape[0],
        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0], _ptr(kv_cache, dt, "kv_cache"),
        _ptr(workspace, None, "workspace"), _nbytes(workspace), _stream(stream)),
        "mla_latent_expand_prepared")


def mla_naive_decode(cfg: MlaConfig, q_nope, q_pe, q_positions, kv_cache, block_table, seq_lens,
                     query_start_loc, workspace, out, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_naive_decode(
        ctypes.byref(cfg), _ptr(q_nope, dt, "q_nope"), _ptr(q_pe, dt, "q_pe"),
        _ptr(q_positions, torch.int32, "q_positions"), _ptr(kv_cache, dt, "kv_cache"),
        kv_cache.shape[0], _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(query_start_loc, torch.int32, "query_start_loc"),
        seq_lens.shape[0], q_nope.shape[0], _ptr(workspace, None, "workspace"), _nbytes(workspace),
        _ptr(out, dt, "out"), _stream(stream)), "mla_naive_decode")


def mla_naive_prefill(cfg: MlaConfig, q_nope, q_pe, q_positions, kv_cache, block_table, seq_lens,
                      query_start_loc, workspace, out, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_naive_prefill(
        ctypes.byref(cfg), _ptr(q_nope, dt, "q_nope"), _ptr(q_pe, dt, "q_pe"),
        _ptr(q_positions, torch.int32, "q_positions"), _ptr(kv_cache, dt, "kv_cache"),
        kv_cache.shape[0], _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(query_start_loc, torch.int32, "query_start_loc"),
        seq_lens.shape[0], q_nope.shape[0], _ptr(workspace, None, "workspace"), _nbytes(workspace),
        _ptr(out, dt, "out"), _stream(stream)), "mla_naive_prefill")


def mla_combine(cfg: MlaConfig, workspace, batch: int, o_lat, stream=None) -> None:
    _check(load().mla_combine(
        ctypes.byref(cfg), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), batch, o_lat.shape[0],
        _ptr(o_lat, torch.float32, "o_lat"), _stream(stream)), "mla_combine")


def mla_combine_out_proj(cfg: MlaConfig, workspace, batch: int, num_q: int, W_uv, out,
                         stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_combine_out_proj(
        ctypes.byref(cfg), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), batch, num_q, _ptr(W_uv, dt, "W_uv"),
        _ptr(out, dt, "out"), _stream(stream)), "mla_combine_out_proj")


def mla_out_proj(cfg: MlaConfig, o_lat, W_uv, out, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_out_proj(
        ctypes.byref(cfg), _ptr(o_lat, torch.float32, "o_lat"), _ptr(W_uv, dt, "W_uv"),
        _ptr(out, dt, "out"), o_lat.shape[0], _stream(stream)), "mla_out_proj")


def mla_proj_workspace_size(cfg: MlaConfig, num_tokens: int, hidden_size: int) -> int:
    return int(load().mla_proj_workspace_size(ctypes.byref(cfg), num_tokens, hidden_size))


def mla_q_proj(cfg: MlaConfig, hidden, W_q, q_nope, q_pe, workspace, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_q_proj(
        ctypes.byref(cfg), _ptr(hidden, dt, "hidden"), _ptr(W_q, dt, "W_q"),
        _ptr(q_nope, dt, "q_nope"), _ptr(q_pe, dt, "q_pe"), hidden.shape[0], hidden.shape[1],
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "mla_q_proj")


def mla_kv_a_proj(cfg: MlaConfig, hidden, W_kv_a, c_kv, k_pe, workspace, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_kv_a_proj(
        ctypes.byref(cfg), _ptr(hidden, dt, "hidden"), _ptr(W_kv_a, dt, "W_kv_a"),
        _ptr(c_kv, dt, "c_kv"), _ptr(k_pe, dt, "k_pe"), hidden.shape[0], hidden.shape[1],
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "mla_kv_a_proj")


def mla_o_proj(cfg: MlaConfig, attn_out, W_o, y, workspace, stream=None) -> None:
    dt = _torch_dtype(cfg)
    _check(load().mla_o_proj(
        ctypes.byref(cfg), _ptr(attn_out, dt, "attn_out"), _ptr(W_o, dt, "W_o"),
        _ptr(y, dt, "y"), attn_out.shape[0], y.shape[1],
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "mla_o_proj")


def mla_get_device_status(status_word, clear: bool = True, stream=None):
    """Returns (status, raw bits)."""
    mask = ctypes.c_uint32(0)
    s = load().mla_get_device_status(_ptr(status_word, None, "status_word"), ctypes.byref(mask),
                                     int(clear), _stream(stream))
    return int(s), int(mask.value)


def mla_selftest_wait_timeout(status_word, timeout_ns: int, stream=None) -> None:
    _check(load().mla_selftest_wait_timeout(_ptr(status_word, None, "status_word"), timeout_ns,
                                            _stream(stream)), "mla_selftest_wait_timeout")
