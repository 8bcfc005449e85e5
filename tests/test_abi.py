"""The C ABI library: it loads, exports every function include/gdn.h declares,
and rejects bad calls on the host before any launch (no GPU needed: the
rejected calls never touch device memory)."""
import ctypes
import os
import re

import torch

import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    lib = gdn.load_library()
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
        assert n in gdn.__all__, f"binding lacks {n}"


def test_status_strings_and_version():
    for code in gdn.STATUS:
        assert gdn.gdn_status_string(code)
    assert gdn.gdn_version() >= 100


def _fake(n=1):
    # Never dereferenced: every call below fails validation first.
    return ctypes.c_void_p(0x10000)


def _prefill(shape, pool_pages=8, start_host=None, init_host=None, block_table=True):
    lib = gdn.load_library()
    desc = gdn.make_desc(shape)
    pool = gdn._Pool(0x100000, shape.page, pool_pages, 0)
    sph, k1 = gdn._host(start_host, torch.int64, "")
    iph, k2 = gdn._host(init_host, torch.int32, "")
    a = gdn._PrefillArgs(len(start_host or [0]), 4, 64, 0, 0x10000, 0x10000, sph, iph, 0x10000, 0x10000,
                         0x10000, 0x10000, 0x10000, 0x10000 if block_table else None, 0x10000, 0x10000, 0x10000)
    return lib.gdn_prefill_chunked(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(a), 0x10000, 1 << 40, None)


def test_prefill_fails_closed_on_off_boundary_resume():
    sh = inputs.TINY
    assert _prefill(sh, start_host=[100], init_host=[3]) == gdn.STATUS_CODE["GDN_ERR_NOT_BLOCK_ALIGNED"]
    # cold start must begin at 0; a resume at 0 is not a resume
    assert _prefill(sh, start_host=[64], init_host=[-1]) == gdn.STATUS_CODE["GDN_ERR_NOT_BLOCK_ALIGNED"]
    assert _prefill(sh, start_host=[0], init_host=[2]) == gdn.STATUS_CODE["GDN_ERR_NOT_BLOCK_ALIGNED"]
    assert _prefill(sh, start_host=[64], init_host=[99]) == gdn.STATUS_CODE["GDN_ERR_PAGE_RANGE"]


def test_prefill_rejects_unsupported_shapes():
    bad = [inputs.with_(inputs.TINY, head_dim_k=48, head_dim_v=48),
           inputs.with_(inputs.TINY, head_dim_k=32, head_dim_v=64),
           inputs.with_(inputs.TINY, chunk_size=24),
           inputs.with_(inputs.TINY, block_size=72),
           inputs.with_(inputs.TINY, in_dtype=inputs.BF16, out_dtype=inputs.F32),
           inputs.with_(inputs.TINY, num_qk_heads=3, num_v_heads=4)]
    for sh in bad:
        assert _prefill(sh, start_host=[0], init_host=[-1]) == gdn.STATUS_CODE["GDN_ERR_UNSUPPORTED_SHAPE"], sh


def test_pool_too_small_or_misaligned_is_rejected():
    lib = gdn.load_library()
    sh = inputs.TINY
    desc = gdn.make_desc(sh)
    a = gdn._DecodeArgs(1, 0, *([0x10000] * 7))
    small = gdn._Pool(0x100000, 256, 4, 0)
    assert lib.gdn_decode_step(ctypes.byref(desc), ctypes.byref(small), ctypes.byref(a), None) == 1
    odd = gdn._Pool(0x100010, sh.page, 4, 0)
    assert lib.gdn_decode_step(ctypes.byref(desc), ctypes.byref(odd), ctypes.byref(a), None) == 1


def test_workspace_is_required_and_sized():
    # the tensor-core prefill (d 128, bf16, block a multiple of 64): the chunk
    # kernel's images for floor(T / 64) + N + 1 chunk slots, per slot T, P,
    # K^T diag(dec), v and the gates of every value head and [K^; Q^] of every
    # qk head (v's image is written only when the chain's levels overlap the
    # chunk kernel; the workspace holds it for every call)
    for sh in (inputs.QWEN27B, inputs.QWEN4B):
        per_slot = sh.num_v_heads * (16384 + 16384 + 32768 + 32768 + 1024) + sh.num_qk_heads * 65536
        for N, T in ((4, 4 * 8192), (1, 229376), (3, 1000), (1, 0)):
            assert gdn.gdn_prefill_workspace_size(sh, N, T) == (T // 64 + N + 1) * per_slot + 1024
            # the packed core: its rows' gates (256-byte rounded) first, then the same images
            # and its fp32 outputs before the gated norm
            gates = -(-(2 * 4 * T * sh.num_v_heads) // 256) * 256
            outs = T * sh.num_v_heads * 128 * 4
            assert gdn.gdn_core_prefill_workspace_size(sh, N, T) == gates + (T // 64 + N + 1) * per_slot + outs + 1024
    # the conv pre-pass path: SiLU(conv) rows in fp32 plus norm factors and gates
    for sh in (inputs.with_(inputs.QWEN27B, head_dim_k=64, head_dim_v=64),
               inputs.with_(inputs.QWEN27B, block_size=784),
               inputs.with_(inputs.QWEN27B, in_dtype=inputs.F32, out_dtype=inputs.F32)):
        need = gdn.gdn_prefill_workspace_size(sh, 4, 4 * 8192)
        assert need >= 4 * 8192 * (sh.conv_dim + 2 * sh.num_qk_heads + 2 * sh.num_v_heads) * 4
        assert need % 256 == 0
    assert gdn.gdn_replay_workspace_size(inputs.QWEN4B, 16) >= 16 * 32 * inputs.QWEN4B.conv_dim * 4
    lib = gdn.load_library()
    desc = gdn.make_desc(inputs.TINY)
    pool = gdn._Pool(0x100000, inputs.TINY.page, 8, 0)
    # host-side arrays stay NULL: only device pointers are faked here
    a = gdn._PrefillArgs(1, 4, 64, 0, 0x10000, 0x10000, None, None, *([0x10000] * 9))
    st = lib.gdn_prefill_chunked(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(a), 0x10000, 16, None)
    assert st == gdn.STATUS_CODE["GDN_ERR_WORKSPACE"]


def test_checkpoint_copy_fails_closed_off_boundary():
    lib = gdn.load_library()
    sh = inputs.TINY
    desc = gdn.make_desc(sh)
    pool = gdn._Pool(0x100000, sh.page, 8, 0)
    nc = (ctypes.c_int64 * 2)(64, 100)
    for fn in (lib.gdn_checkpoint_resume, lib.gdn_checkpoint_save):
        st = fn(ctypes.byref(desc), ctypes.byref(pool), 0x10000, 0x10000, nc, 2, 0x10000, None)
        assert st == gdn.STATUS_CODE["GDN_ERR_NOT_BLOCK_ALIGNED"]


def test_replay_rejects_oversized_append_and_bad_rollback_args():
    lib = gdn.load_library()
    sh = inputs.TINY
    desc = gdn.make_desc(sh)
    pool = gdn._Pool(0x100000, sh.page, 8, 0)
    a = gdn._ReplayArgs(2, 33, *([0x10000] * 11), 0x10000, 1 << 40)
    assert lib.gdn_replay_append(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(a), None) == \
        gdn.STATUS_CODE["GDN_ERR_LOG_OVERFLOW"]
    assert lib.gdn_replay_rollback(0x10000, 0x10000, 40, 2, 0x10000, None) == gdn.STATUS_CODE["GDN_ERR_INVALID_ARG"]


def test_flush_boundary_checkpoint_host_checks():
    """Boundary checkpoints need both arrays and the tensor-core shape; the
    checks run before any launch (the device pointers are fake)."""
    lib = gdn.load_library()
    F = 0x10000
    for sh, bpage, want in ((inputs.QWEN4B, None, "GDN_ERR_INVALID_ARG"),
                            (inputs.TINY, F, "GDN_ERR_UNSUPPORTED_SHAPE")):
        desc = gdn.make_desc(sh)
        pool = gdn._Pool(0x100000, sh.page, 8, 0)
        r = gdn._ReplayArgs(2, 0, *([F] * 11), F, 1 << 40, F, bpage)
        assert lib.gdn_replay_flush(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(r), None) == \
            gdn.STATUS_CODE[want], sh


def test_empty_batches_are_no_ops():
    lib = gdn.load_library()
    sh = inputs.TINY
    desc = gdn.make_desc(sh)
    pool = gdn._Pool(0x100000, sh.page, 8, 0)
    a = gdn._DecodeArgs(0, 0, *([None] * 7))
    assert lib.gdn_decode_step(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(a), None) == 0
    r = gdn._ReplayArgs(0, 0, *([None] * 11), None, 0)
    assert lib.gdn_replay_flush(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(r), None) == 0
    assert lib.gdn_replay_rollback(None, None, 4, 0, None, None) == 0


def test_mixed_step_host_checks():
    """gdn_mixed_step validates its host arrays before launching anything
    (device pointers here are fake and never dereferenced)."""
    lib = gdn.load_library()
    sh = inputs.TINY
    desc = gdn.make_desc(sh)
    pool = gdn._Pool(0x100000, sh.page, 8, 0)
    F = 0x10000

    # every case below fails a host check, so nothing is launched on the fake pointers
    def call(cu, dec, sp=None, ip=None, drop_dec_host=False, total=None):
        cu_h = (ctypes.c_int32 * len(cu))(*cu)
        dec_h = (ctypes.c_int8 * len(dec))(*dec)
        sp_h = (ctypes.c_int64 * len(sp))(*sp) if sp is not None else None
        ip_h = (ctypes.c_int32 * len(ip))(*ip) if ip is not None else None
        n = len(dec)
        a = gdn._MixedArgs(n, 2, cu[-1] if total is None else total, 0, F, ctypes.addressof(cu_h), F,
                           None if drop_dec_host else ctypes.addressof(dec_h), F,
                           ctypes.addressof(sp_h) if sp_h is not None else None, F,
                           ctypes.addressof(ip_h) if ip_h is not None else None, F, F, F, F, F, F, F, F)
        return lib.gdn_mixed_step(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(a), F, 1 << 40, None)

    code = gdn.STATUS_CODE
    assert call([0, 2, 3], [1, 0]) == code["GDN_ERR_INVALID_ARG"]          # a decode entry of two rows
    assert call([0, 1, 3], [1, 0], drop_dec_host=True) == code["GDN_ERR_INVALID_ARG"]
    assert call([0, 1, 3], [1, 0], sp=[0, 10], ip=[-1, 2]) == code["GDN_ERR_NOT_BLOCK_ALIGNED"]
    assert call([0, 1, 3], [1, 0], sp=[0, 64], ip=[-1, 9]) == code["GDN_ERR_PAGE_RANGE"]
    assert call([0, 1, 4], [1, 0], total=5) == code["GDN_ERR_INVALID_ARG"]  # cu_seqlens end != total
    a = gdn._MixedArgs(0, 0, 0, 0, *([None] * 16))
    assert lib.gdn_mixed_step(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(a), None, 0, None) == 0


def test_core_prefill_needs_the_tensor_core_path():
    """The packed prefill's gated norm lives in the tensor-core kernel's
    epilogue: other shapes are refused before anything launches."""
    lib = gdn.load_library()
    sh = inputs.LayerShape(2, 4, 64, 64, 64, 16)
    desc = gdn.make_desc(sh)
    pool = gdn._Pool(0x100000, sh.page, 8, 0)
    F = 0x10000
    a = gdn._PrefillArgs(1, 1, 64, 0, F, F, None, None, F, None, None, F, F, F, F, F, F)
    c = gdn._CoreArgs(F, F, F, F, 1e-6, 0)
    st = lib.gdn_core_prefill(ctypes.byref(desc), ctypes.byref(pool), ctypes.byref(a), ctypes.byref(c), F,
                              1 << 40, None)
    assert st == gdn.STATUS_CODE["GDN_ERR_UNSUPPORTED_SHAPE"]
