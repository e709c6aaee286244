"""Python binding of ``libmla.so`` -- MLA decode with matrix absorption on B300.

The functions here carry the C ABI's names (``include/mla.h``) and only
marshal arguments: tensors become raw device pointers, the stream becomes a
``cudaStream_t``, and a non-``MLA_OK`` status raises :class:`MLAError`.
Every step of the path runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback.  Importing this package fails loudly when the library
has not been built (``python mla_latent_kv_74_b300/build.py``).

Example (one decode step, all tensors on ``cuda``)::

    import mla_latent_kv_74_b300 as mla
    dims = mla.Dims(H=128, d_h=128, d_c=512, d_r=64, block_size=64)
    mla.mla_append_cache(cache, num_blocks, block_table, seqlens, c_kv, k_r, dims)
    mla.mla_absorb_query(q_nope, W_UK, q_lat, dims)
    ws = mla.alloc_workspace(B, Hq, max_seqlen, dims)
    mla.mla_decode(q_lat, q_rope, cache, num_blocks, block_table, seqlens,
                   max_seqlen, dims, o_lat, lse, ws)
    mla.mla_out_proj(o_lat, W_UV, out, dims)
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_BOUNDS = 5
MLA_ERR_TIMEOUT = 6
MLA_BF16 = 0
MLA_FP32 = 1

# every symbol include/mla.h and include/mla_debug.h declare
EXPORTED = (
    "mla_absorb_query",
    "mla_append_cache",
    "mla_decode_workspace_size",
    "mla_decode",
    "mla_decode_blocks",
    "mla_combine_pieces",
    "mla_out_proj",
    "mla_get_error",
    "mla_status_string",
    "mla_decode_noalloc",
    "mla_decode_noalloc_get_error",
    "mla_project_append_workspace_size",
    "mla_project_append",
    "mla_o_proj_workspace_size",
    "mla_o_proj",
    "mla_project_query_workspace_size",
    "mla_project_query",
    "mla_prefill_workspace_size",
    "mla_prefill",
    "mla_selftest_lost_wait",
    "mla_debug_set_decode_pairs",
)

# size of the scratch array built into the library for mla_decode_noalloc
NOALLOC_SCRATCH_BYTES = 48 << 20


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class Dims(ctypes.Structure):
    """``mla_dims``: H, d_h, d_c, d_r, block_size, dtype, scale (0 = 1/sqrt(d_h+d_r))."""

    _fields_ = [("H", ctypes.c_int), ("d_h", ctypes.c_int), ("d_c", ctypes.c_int),
                ("d_r", ctypes.c_int), ("block_size", ctypes.c_int), ("dtype", ctypes.c_int),
                ("scale", ctypes.c_float)]

    def __init__(self, H, d_h, d_c, d_r, block_size=64, dtype=MLA_BF16, scale=0.0):
        if isinstance(dtype, torch.dtype):
            dtype = MLA_BF16 if dtype == torch.bfloat16 else MLA_FP32
        super().__init__(H, d_h, d_c, d_r, block_size, dtype, scale)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == MLA_BF16 else torch.float32


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python mla_latent_kv_74_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D = ctypes.POINTER(Dims)
    sig = {
        "mla_absorb_query": [P, P, P, I, I, D, P],
        "mla_append_cache": [P, I, P, I, P, P, P, I, I, D, P],
        "mla_decode_workspace_size": [I, I, I, D, ctypes.POINTER(Z)],
        "mla_decode": [P, P, P, I, P, I, P, I, I, I, D, P, P, P, Z, P],
        "mla_decode_blocks": [P, P, P, I, P, I, P, I, I, I, I, I, D, P, P, P, Z, P],
        "mla_combine_pieces": [P, P, I, I, I, D, P, P, P],
        "mla_out_proj": [P, P, P, I, I, D, P],
        "mla_get_error": [P, P],
        "mla_status_string": [I],
        "mla_decode_noalloc": [P, P, P, I, P, I, P, I, I, I, D, P, P, P],
        "mla_decode_noalloc_get_error": [P],
        "mla_project_append_workspace_size": [I, I, I, D, ctypes.POINTER(Z)],
        "mla_project_append": [P, P, P, I, ctypes.c_float, P, I, P, I, P, I, I, D, P, Z, P],
        "mla_o_proj_workspace_size": [I, I, I, D, ctypes.POINTER(Z)],
        "mla_o_proj": [P, P, P, I, I, I, D, P, Z, P],
        "mla_project_query_workspace_size": [I, I, I, D, ctypes.POINTER(Z)],
        "mla_project_query": [P, P, P, I, ctypes.c_float, P, I, I, D, P, P, P, Z, P],
        "mla_prefill_workspace_size": [I, D, ctypes.POINTER(Z)],
        "mla_prefill": [P, P, P, P, P, P, P, I, I, I, D, P, P, P, Z, P],
        "mla_selftest_lost_wait": [P, P],
        "mla_debug_set_decode_pairs": [I],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "mla_status_string" else ctypes.c_int
    return lib


_lib = _load()


def status_string(status: int) -> str:
    return _lib.mla_status_string(int(status)).decode()


def _ptr(t):
    """Raw device pointer of a tensor; the library reads dense row-major
    memory, so strided views are refused rather than misread."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(t.shape)} with strides {t.stride()} is not "
                         "contiguous; pass .contiguous()")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != MLA_OK:
        raise MLAError(status, where)


def mla_absorb_query(q_nope, W_UK, q_lat, dims: Dims, stream=None):
    """``q_lat = W_UK^T q_nope`` per head; shapes [B,Hq,H,d_h] -> [B,Hq,H,d_c]."""
    B, Hq = q_nope.shape[0], q_nope.shape[1]
    _check(_lib.mla_absorb_query(_ptr(q_nope), _ptr(W_UK), _ptr(q_lat), B, Hq,
                                 ctypes.byref(dims), _stream(stream)), "mla_absorb_query")


def mla_append_cache(cache, num_blocks, block_table, seqlens, c_kv, k_r, dims: Dims,
                     stream=None):
    """Write ``[c_kv ; k_r]`` of the ``n_new`` newest tokens into the paged cache."""
    B, n_new = c_kv.shape[0], c_kv.shape[1]
    _check(_lib.mla_append_cache(_ptr(cache), int(num_blocks), _ptr(block_table),
                                 block_table.shape[1], _ptr(seqlens), _ptr(c_kv), _ptr(k_r),
                                 B, n_new, ctypes.byref(dims), _stream(stream)),
           "mla_append_cache")


def mla_project_append_workspace_size(B, n_new, d_model, dims: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mla_project_append_workspace_size(B, n_new, int(d_model), ctypes.byref(dims),
                                                  ctypes.byref(n)),
           "mla_project_append_workspace_size")
    return n.value


def mla_project_append(h, W_DKV, W_KR, cache, num_blocks, block_table, seqlens, dims: Dims,
                       workspace, rope_base=10000.0, stream=None):
    """``[W_DKV h ; RoPE(W_KR h, p)]`` of the ``n_new`` newest tokens, written
    into the paged cache; ``h`` is [B, n_new, d_model]."""
    B, n_new, d_model = h.shape
    _check(_lib.mla_project_append(_ptr(h), _ptr(W_DKV), _ptr(W_KR), int(d_model),
                                   float(rope_base), _ptr(cache), int(num_blocks),
                                   _ptr(block_table), block_table.shape[1], _ptr(seqlens),
                                   B, n_new, ctypes.byref(dims), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(),
                                   _stream(stream)),
           "mla_project_append")


def mla_project_query_workspace_size(B, Hq, d_model, dims: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mla_project_query_workspace_size(B, Hq, int(d_model), ctypes.byref(dims),
                                                 ctypes.byref(n)),
           "mla_project_query_workspace_size")
    return n.value


def mla_project_query(h, W_Q, W_QR, seqlens, dims: Dims, q_nope, q_rope, workspace,
                      rope_base=10000.0, stream=None):
    """``q_nope = W_Q h``, ``q_rope = RoPE(W_QR h, p)`` per head; ``h`` [B,Hq,d_model]."""
    B, Hq, d_model = h.shape
    _check(_lib.mla_project_query(_ptr(h), _ptr(W_Q), _ptr(W_QR), int(d_model),
                                  float(rope_base), _ptr(seqlens), B, Hq, ctypes.byref(dims),
                                  _ptr(q_nope), _ptr(q_rope), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  _stream(stream)),
           "mla_project_query")


def mla_o_proj_workspace_size(B, Hq, d_model, dims: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mla_o_proj_workspace_size(B, Hq, int(d_model), ctypes.byref(dims),
                                          ctypes.byref(n)), "mla_o_proj_workspace_size")
    return n.value


def mla_o_proj(out, W_O, u, dims: Dims, workspace, stream=None):
    """``u = W_O [out_0; ..; out_{H-1}]`` per row; out [B,Hq,H,d_h] -> u [B,Hq,d_model]."""
    B, Hq = out.shape[0], out.shape[1]
    _check(_lib.mla_o_proj(_ptr(out), _ptr(W_O), _ptr(u), B, Hq, int(W_O.shape[0]),
                           ctypes.byref(dims), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream)),
           "mla_o_proj")


def mla_decode_workspace_size(B, Hq, max_seqlen, dims: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mla_decode_workspace_size(B, Hq, int(max_seqlen), ctypes.byref(dims),
                                          ctypes.byref(n)), "mla_decode_workspace_size")
    return n.value


def alloc_workspace(B, Hq, max_seqlen, dims: Dims, device="cuda"):
    """A zero-filled workspace of the size ``mla_decode`` needs (torch-owned)."""
    n = mla_decode_workspace_size(B, Hq, max_seqlen, dims)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def mla_decode(q_lat, q_rope, cache, num_blocks, block_table, seqlens, max_seqlen,
               dims: Dims, o_lat, lse, workspace, stream=None):
    """Absorbed MLA decode: ``o_lat = softmax(scores) C``, ``lse`` per row."""
    B, Hq = q_lat.shape[0], q_lat.shape[1]
    _check(_lib.mla_decode(_ptr(q_lat), _ptr(q_rope), _ptr(cache), int(num_blocks),
                           _ptr(block_table), block_table.shape[1], _ptr(seqlens),
                           int(max_seqlen), B, Hq, ctypes.byref(dims), _ptr(o_lat), _ptr(lse),
                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream)), "mla_decode")


def mla_decode_blocks(q_lat, q_rope, cache, num_blocks, block_table, seqlens, max_seqlen,
                      first_block, end_block, dims: Dims, o_lat, lse, workspace, stream=None):
    """``mla_decode`` over the cache blocks ``[first_block, end_block)`` of every
    sequence: one split-KV piece (``o_lat``, ``lse`` over those keys alone)."""
    B, Hq = q_lat.shape[0], q_lat.shape[1]
    _check(_lib.mla_decode_blocks(_ptr(q_lat), _ptr(q_rope), _ptr(cache), int(num_blocks),
                                  _ptr(block_table), block_table.shape[1], _ptr(seqlens),
                                  int(max_seqlen), B, Hq, int(first_block), int(end_block),
                                  ctypes.byref(dims), _ptr(o_lat), _ptr(lse), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "mla_decode_blocks")


def mla_combine_pieces(o_pieces, lse_pieces, dims: Dims, o_lat, lse, stream=None):
    """Merge ``P`` stacked pieces ``[P,B,Hq,H,d_c]`` / ``[P,B,Hq,H]`` (outputs of
    ``mla_decode_blocks`` over disjoint ranges) into ``o_lat`` and ``lse``."""
    P, B, Hq = o_pieces.shape[0], o_pieces.shape[1], o_pieces.shape[2]
    _check(_lib.mla_combine_pieces(_ptr(o_pieces), _ptr(lse_pieces), P, B, Hq,
                                   ctypes.byref(dims), _ptr(o_lat), _ptr(lse), _stream(stream)),
           "mla_combine_pieces")


def mla_out_proj(o_lat, W_UV, out, dims: Dims, stream=None):
    """``out = W_UV o_lat`` per head; shapes [B,Hq,H,d_c] -> [B,Hq,H,d_h]."""
    B, Hq = o_lat.shape[0], o_lat.shape[1]
    _check(_lib.mla_out_proj(_ptr(o_lat), _ptr(W_UV), _ptr(out), B, Hq, ctypes.byref(dims),
                             _stream(stream)), "mla_out_proj")


def mla_decode_noalloc(q_lat, q_rope, cache, num_blocks, block_table, seqlens, max_seqlen,
                       dims: Dims, o_lat, lse, stream=None):
    """``mla_decode`` without a caller-provided workspace: the library uses
    its built-in scratch array (for callers that cannot allocate device
    memory).  Calls share that array, so order them on one stream."""
    B, Hq = q_lat.shape[0], q_lat.shape[1]
    _check(_lib.mla_decode_noalloc(_ptr(q_lat), _ptr(q_rope), _ptr(cache), int(num_blocks),
                                   _ptr(block_table), block_table.shape[1], _ptr(seqlens),
                                   int(max_seqlen), B, Hq, ctypes.byref(dims), _ptr(o_lat),
                                   _ptr(lse), _stream(stream)), "mla_decode_noalloc")


def mla_decode_noalloc_get_error(stream=None) -> int:
    """Synchronise, read and clear the built-in array's device error word
    (the errors of ``mla_decode_noalloc``); returns the status."""
    return int(_lib.mla_decode_noalloc_get_error(_stream(stream)))


def mla_prefill_workspace_size(total_tokens, dims: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mla_prefill_workspace_size(int(total_tokens), ctypes.byref(dims),
                                           ctypes.byref(n)), "mla_prefill_workspace_size")
    return n.value


def mla_prefill(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, cu_seqlens, max_seqlen, dims: Dims,
                out, lse, workspace, stream=None):
    """Causal MLA prefill of packed sequences in the standard order (K and V
    rebuilt from the latents, attention over d_h + d_r and d_h):
    q_nope [T,H,d_h], q_rope [T,H,d_r], c_kv [T,d_c], k_r [T,d_r],
    cu_seqlens [B+1] int32 on the device -> out [T,H,d_h], lse [T,H]."""
    _check(_lib.mla_prefill(_ptr(q_nope), _ptr(q_rope), _ptr(c_kv), _ptr(k_r), _ptr(W_UK),
                            _ptr(W_UV), _ptr(cu_seqlens), cu_seqlens.shape[0] - 1,
                            int(max_seqlen), q_nope.shape[0], ctypes.byref(dims), _ptr(out),
                            _ptr(lse), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream)),
           "mla_prefill")


def mla_selftest_lost_wait(workspace, stream=None):
    """Launch the failure-path self-test: a bounded wait that nothing
    satisfies expires (after 2 s) and records MLA_ERR_TIMEOUT in
    ``workspace``'s error word (read it with ``mla_get_error``)."""
    _check(_lib.mla_selftest_lost_wait(_ptr(workspace), _stream(stream)),
           "mla_selftest_lost_wait")


def mla_get_error(workspace, stream=None) -> int:
    """Synchronise, read and clear the device error word; returns the status."""
    return int(_lib.mla_get_error(_ptr(workspace), _stream(stream)))


def mla_debug_set_decode_pairs(pairs: int) -> int:
    """Test hook (``include/mla_debug.h``): limit the CTA pairs of the
    tensor-core decode's split plan (0 = no limit); returns the previous
    limit."""
    return int(_lib.mla_debug_set_decode_pairs(int(pairs)))


def raw_lib():
    """The ``ctypes.CDLL`` handle, for callers that pass raw pointers."""
    return _lib
