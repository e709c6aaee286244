"""The C-ABI library loads, exports every symbol ``include/mla.h`` declares,
and rejects bad arguments on the host before launching anything.

These tests make no compute call: every call here fails validation and
returns before touching CUDA, so they run on a machine without a GPU.
"""

import ctypes
import glob
import os
import re

import pytest

import mla_latent_kv_74_b300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for hdr in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        txt = re.sub(r"/\*.*?\*/", "", open(hdr).read(), flags=re.S)
        names |= set(re.findall(r"\b(mla_[a-z_]+)\s*\(", txt))
    return sorted(names)


def test_library_builds_and_loads():
    assert os.path.exists(m.LIB_PATH)
    ctypes.CDLL(m.LIB_PATH)


def test_every_declared_symbol_is_exported():
    declared = _declared_symbols()
    assert set(declared) == set(m.EXPORTED), declared
    lib = ctypes.CDLL(m.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_debug_pairs_limit_round_trips():
    assert m.mla_debug_set_decode_pairs(7) == 0
    assert m.mla_debug_set_decode_pairs(-3) == 7
    assert m.mla_debug_set_decode_pairs(0) == 0


def test_status_strings():
    for code in range(7):
        s = m.status_string(code)
        assert s.startswith("MLA_")
    assert m.status_string(99) == "unknown mla_status"


def _dims(**kw):
    base = dict(H=128, d_h=128, d_c=512, d_r=64, block_size=64, dtype=m.MLA_BF16)
    base.update(kw)
    return m.Dims(**base)


def test_workspace_size_validation():
    lib = m.raw_lib()
    n = ctypes.c_size_t()
    assert lib.mla_decode_workspace_size(4, 1, 100, None, ctypes.byref(n)) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_workspace_size(4, 1, 100, ctypes.byref(_dims(d_c=1024)),
                                         ctypes.byref(n)) == m.MLA_ERR_UNSUPPORTED
    assert lib.mla_decode_workspace_size(4, 0, 100, ctypes.byref(_dims()),
                                         ctypes.byref(n)) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_workspace_size(4, 1, 100, ctypes.byref(_dims()), None) == \
        m.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_workspace_size(64, 1, 8192, ctypes.byref(_dims()),
                                         ctypes.byref(n)) == m.MLA_OK
    assert n.value >= 256


def test_decode_path_limits():
    """The tensor-core decode takes at most 8192 (sequence, slot) items; larger
    batches fall through to the CUDA-core kernel (whose workspace grows with
    the rows), and more than 65535 items are refused before any launch."""
    lib = m.raw_lib()
    n = ctypes.c_size_t()
    d = ctypes.byref(_dims())
    assert lib.mla_decode_workspace_size(8192, 1, 64, d, ctypes.byref(n)) == m.MLA_OK
    tc_bytes = n.value
    assert tc_bytes < 48 << 20  # split partials of 74 CTA pairs, not of the rows
    assert lib.mla_decode_workspace_size(8193, 1, 64, d, ctypes.byref(n)) == m.MLA_OK
    assert n.value > 8193 * 128 * 512 * 4  # one fp32 partial row per (row, split)
    assert lib.mla_decode_workspace_size(65536, 1, 64, d, ctypes.byref(n)) == \
        m.MLA_ERR_UNSUPPORTED
    assert lib.mla_decode_workspace_size(32768, 2, 64, d, ctypes.byref(n)) == \
        m.MLA_ERR_UNSUPPORTED
    ok = ctypes.c_void_p(1 << 20)
    args = [ok, ok, ok, 4, ok, 4, ok, 64, 65536, 1, d, ok, ok, ok, 1 << 40, None]
    assert lib.mla_decode(*args) == m.MLA_ERR_UNSUPPORTED
    assert lib.mla_decode_noalloc(ok, ok, ok, 4, ok, 4, ok, 64, 65536, 1, d, ok, ok,
                                  None) == m.MLA_ERR_UNSUPPORTED


def test_noalloc_fits_every_tensor_core_workload():
    """The built-in array of mla_decode_noalloc holds the workspace of each
    DeepSeek-V2-shaped workload (the ragged two-slot one included), so none of
    them is refused with MLA_ERR_WORKSPACE."""
    lib = m.raw_lib()
    n = ctypes.c_size_t()
    for H, B, Hq, max_seqlen in ((16, 32, 1, 4096), (128, 64, 1, 8192), (128, 128, 2, 32768),
                                 (128, 4, 1, 131072),
                                 # the most items the tensor-core plan takes, with
                                 # few heads (two piece slots per SM) and with pairs
                                 (16, 8192, 1, 64), (128, 4096, 2, 64)):
        assert lib.mla_decode_workspace_size(B, Hq, max_seqlen, ctypes.byref(_dims(H=H)),
                                             ctypes.byref(n)) == m.MLA_OK
        assert n.value <= m.NOALLOC_SCRATCH_BYTES, (H, B, Hq, n.value)


@pytest.mark.parametrize("bad", [dict(H=0), dict(H=300), dict(d_h=256), dict(d_r=65),
                                 dict(block_size=0), dict(dtype=7)])
def test_unsupported_dims_rejected(bad):
    lib = m.raw_lib()
    d = _dims(**bad)
    p = ctypes.c_void_p(256)
    assert lib.mla_absorb_query(p, p, p, 1, 1, ctypes.byref(d), None) == m.MLA_ERR_UNSUPPORTED
    assert lib.mla_out_proj(p, p, p, 1, 1, ctypes.byref(d), None) == m.MLA_ERR_UNSUPPORTED


def test_null_and_misaligned_pointers_rejected():
    lib = m.raw_lib()
    d = ctypes.byref(_dims())
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 2)
    assert lib.mla_absorb_query(None, ok, ok, 1, 1, d, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_absorb_query(ok, mis, ok, 1, 1, d, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_out_proj(ok, ok, mis, 1, 1, d, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_append_cache(ok, 4, ok, 4, ok, ok, None, 1, 1, d, None) == \
        m.MLA_ERR_INVALID_ARG  # k_r missing with d_r > 0
    # decode: cache must be 128-byte aligned, workspace present and large enough
    cache_mis = ctypes.c_void_p((1 << 20) + 64)
    args = [ok, ok, cache_mis, 4, ok, 4, ok, 64, 1, 1, d, ok, ok, ok, 1 << 30, None]
    assert lib.mla_decode(*args) == m.MLA_ERR_INVALID_ARG
    args[2] = ok
    args[13] = None
    assert lib.mla_decode(*args) == m.MLA_ERR_WORKSPACE
    args[13] = ok
    args[14] = 16
    assert lib.mla_decode(*args) == m.MLA_ERR_WORKSPACE
    args[9] = 0  # Hq
    assert lib.mla_decode(*args) == m.MLA_ERR_INVALID_ARG


def test_project_append_host_validation():
    lib = m.raw_lib()
    d = ctypes.byref(_dims())
    n = ctypes.c_size_t()
    F = ctypes.c_float
    assert lib.mla_project_append_workspace_size(64, 1, 5120, d, ctypes.byref(n)) == m.MLA_OK
    # 27 K splits of 3 chunks for d_model = 5120: 27 x 64 tokens x 576 fp32
    assert n.value == 27 * 64 * 576 * 4
    assert lib.mla_project_append_workspace_size(64, 1, 5000, d, ctypes.byref(n)) == \
        m.MLA_ERR_UNSUPPORTED  # d_model not a multiple of 64
    assert lib.mla_project_append_workspace_size(
        1, 1, 512, ctypes.byref(_dims(dtype=m.MLA_FP32)), ctypes.byref(n)) == m.MLA_ERR_UNSUPPORTED
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 2)
    args = [ok, ok, ok, 512, F(10000.0), ok, 4, ok, 4, ok, 1, 1, d, ok, 1 << 30, None]
    bad = list(args); bad[1] = mis
    assert lib.mla_project_append(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args); bad[4] = F(0.0)
    assert lib.mla_project_append(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args); bad[14] = 16
    assert lib.mla_project_append(*bad) == m.MLA_ERR_WORKSPACE
    bad = list(args); bad[13] = None
    assert lib.mla_project_append(*bad) == m.MLA_ERR_WORKSPACE
    bad = list(args); bad[3] = 100
    assert lib.mla_project_append(*bad) == m.MLA_ERR_UNSUPPORTED
    empty = list(args); empty[10] = 0
    assert lib.mla_project_append(*empty) == m.MLA_OK


def test_o_proj_host_validation():
    lib = m.raw_lib()
    d = ctypes.byref(_dims())
    n = ctypes.c_size_t()
    assert lib.mla_o_proj_workspace_size(64, 1, 5120, d, ctypes.byref(n)) == m.MLA_OK
    # K = 128 heads x 128 = 256 chunks of 64, 40 M tiles: 7 splits of 37 chunks
    assert n.value == 7 * 64 * 5120 * 4
    assert lib.mla_o_proj_workspace_size(64, 1, 5121, d, ctypes.byref(n)) == m.MLA_ERR_UNSUPPORTED
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    args = [ok, ok, ok, 4, 1, 5120, d, ok, 1 << 30, None]
    bad = list(args); bad[2] = mis
    assert lib.mla_o_proj(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args); bad[8] = 64
    assert lib.mla_o_proj(*bad) == m.MLA_ERR_WORKSPACE
    bad = list(args); bad[4] = 0
    assert lib.mla_o_proj(*bad) == m.MLA_ERR_INVALID_ARG
    empty = list(args); empty[3] = 0
    assert lib.mla_o_proj(*empty) == m.MLA_OK


def test_project_query_host_validation():
    lib = m.raw_lib()
    d = ctypes.byref(_dims())
    n = ctypes.c_size_t()
    F = ctypes.c_float
    assert lib.mla_project_query_workspace_size(64, 1, 5120, d, ctypes.byref(n)) == m.MLA_OK
    # 128 + 64 M tiles, 80 K chunks: three splits of 27 chunks (two waves of
    # 296 CTAs beat one slow wave), 64 rows x 128 heads x (128 + 64) fp32 each
    assert n.value == 3 * 64 * 128 * 192 * 4
    assert lib.mla_project_query_workspace_size(64, 1, 5000, d, ctypes.byref(n)) == \
        m.MLA_ERR_UNSUPPORTED
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    args = [ok, ok, ok, 512, F(10000.0), ok, 2, 1, d, ok, ok, ok, 1 << 30, None]
    bad = list(args); bad[10] = mis
    assert lib.mla_project_query(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args); bad[12] = 16
    assert lib.mla_project_query(*bad) == m.MLA_ERR_WORKSPACE
    bad = list(args); bad[4] = F(-1.0)
    assert lib.mla_project_query(*bad) == m.MLA_ERR_INVALID_ARG
    empty = list(args); empty[6] = 0
    assert lib.mla_project_query(*empty) == m.MLA_OK


def test_prefill_host_validation():
    lib = m.raw_lib()
    d = ctypes.byref(_dims())
    n = ctypes.c_size_t()
    assert lib.mla_prefill_workspace_size(4096, d, ctypes.byref(n)) == m.MLA_OK
    # error-word header plus [K_nope | V] in bf16 per (token, head)
    assert n.value == 256 + 4096 * 128 * 256 * 2
    assert lib.mla_prefill_workspace_size(-1, d, ctypes.byref(n)) == m.MLA_ERR_INVALID_ARG
    bad_dims = ctypes.byref(m.Dims(128, 128, 512, 32))
    assert lib.mla_prefill_workspace_size(16, bad_dims, ctypes.byref(n)) == m.MLA_ERR_UNSUPPORTED
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    args = [ok, ok, ok, ok, ok, ok, ok, 2, 300, 500, d, ok, ok, ok, 1 << 30, None]
    for i in (0, 1, 2, 3, 4, 5, 11):  # tensors must be 16-byte aligned
        bad = list(args); bad[i] = mis
        assert lib.mla_prefill(*bad) == m.MLA_ERR_INVALID_ARG, i
    bad = list(args); bad[6] = None
    assert lib.mla_prefill(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args); bad[14] = 1 << 20
    assert lib.mla_prefill(*bad) == m.MLA_ERR_WORKSPACE
    bad = list(args); bad[13] = mis
    assert lib.mla_prefill(*bad) == m.MLA_ERR_WORKSPACE
    bad = list(args); bad[7] = 70000
    assert lib.mla_prefill(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args); bad[10] = bad_dims
    assert lib.mla_prefill(*bad) == m.MLA_ERR_UNSUPPORTED
    for i in (7, 9):  # no sequences or no tokens: nothing to do
        empty = list(args); empty[i] = 0
        assert lib.mla_prefill(*empty) == m.MLA_OK
    bad = list(args); bad[8] = 0  # tokens, but no sequence may hold one
    assert lib.mla_prefill(*bad) == m.MLA_ERR_INVALID_ARG


def test_empty_batch_is_a_noop():
    lib = m.raw_lib()
    d = ctypes.byref(_dims())
    assert lib.mla_absorb_query(None, None, None, 0, 1, d, None) == m.MLA_OK
    assert lib.mla_out_proj(None, None, None, 0, 1, d, None) == m.MLA_OK
    assert lib.mla_append_cache(None, 1, None, 1, None, None, None, 0, 1, d, None) == m.MLA_OK
    assert lib.mla_decode(None, None, None, 1, None, 1, None, 0, 0, 1, d, None, None, None, 0,
                          None) == m.MLA_OK


def test_strided_tensor_refused():
    """A strided view would be read as dense memory: the binding refuses it."""
    import torch
    t = torch.zeros(4, 8).t()
    with pytest.raises(ValueError):
        m._ptr(t)
    x = torch.zeros(4, 8)
    assert m._ptr(x) == x.data_ptr()


def test_block_range_and_combine_validation():
    """mla_decode_blocks refuses a negative or reversed block range and the
    shapes only the CUDA-core path takes; mla_combine_pieces refuses P < 1,
    missing or misaligned pointers and non-tensor-core shapes.  All of it is
    decided on the host, before anything is launched."""
    lib = m.raw_lib()
    d = ctypes.byref(_dims())
    ok = ctypes.c_void_p(1 << 20)

    def blocks(first, end, dims=d, B=2):
        return lib.mla_decode_blocks(ok, ok, ok, 4, ok, 4, ok, 64, B, 1, first, end, dims, ok,
                                     ok, ok, 1 << 40, None)

    assert blocks(-1, 3) == m.MLA_ERR_INVALID_ARG
    assert blocks(3, 2) == m.MLA_ERR_INVALID_ARG
    assert blocks(0, 3, B=0) == m.MLA_OK  # nothing to do
    fp32 = ctypes.byref(m.Dims(H=4, d_h=16, d_c=16, d_r=8, block_size=32, dtype=m.MLA_FP32))
    assert blocks(0, 3, dims=fp32) == m.MLA_ERR_UNSUPPORTED  # CUDA-core shapes
    assert lib.mla_combine_pieces(ok, ok, 0, 2, 1, d, ok, ok, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_combine_pieces(None, ok, 2, 2, 1, d, ok, ok, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_combine_pieces(ctypes.c_void_p((1 << 20) + 2), ok, 2, 2, 1, d, ok, ok,
                                  None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_combine_pieces(ok, ok, 2, 2, 1, fp32, ok, ok, None) == \
        m.MLA_ERR_UNSUPPORTED
    assert lib.mla_combine_pieces(ok, ok, 2, 0, 1, d, ok, ok, None) == m.MLA_OK
