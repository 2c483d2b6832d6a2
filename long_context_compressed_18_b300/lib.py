"""Python binding of the C ABI in ``include/csa.h``.

Argument marshalling only: each function passes tensor data pointers, sizes
and the current CUDA stream to the function of the same name in
``libcsa_b300.so`` and raises :class:`CsaError` on a non-OK status.  Every
step of the path runs in the library's kernels; there is no fallback -- if
the shared library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libcsa_b300.so")

F32, BF16, E4M3, E2M1 = 0, 1, 2, 3
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "ALIGNMENT", 4: "WORKSPACE",
          5: "CUDA", 6: "TIMEOUT", 7: "DEVICE"}

EXPORTS = ("csa_compress", "csa_compress_per_channel", "csa_index_scores_workspace_size", "csa_index_scores",
           "csa_topk_select_workspace_size", "csa_topk_select", "csa_topk_select_noalloc",
           "csa_index_topk_workspace_size",
           "csa_index_topk", "csa_index_topk_varlen", "csa_decode_append", "csa_sparse_attn_workspace_size", "csa_sparse_attn", "hca_attn",
           "swa_attn", "csa_device_status", "csa_last_error", "csa_wait_selftest")


class CsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None
_P, _I, _L, _S, _F = C.c_void_p, C.c_int, C.c_int64, C.c_size_t, C.c_float


def load():
    """Load the library (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OSError(f"{LIB_PATH} is missing: build it with long_context_compressed_18_b300.build")
    lib = C.CDLL(LIB_PATH)
    sig = {
        "csa_compress": ([_I, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _P], _I),
        "csa_compress_per_channel": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
        "csa_index_scores_workspace_size": ([_I, _I, _I, _I], _S),
        "csa_index_scores": ([_I, _I, _L, _I, _I, _I, _I, _P, _I, _P, _P, _I, _P, _P, _I, _P, _I, _P, _S, _P], _I),
        "csa_topk_select_workspace_size": ([_I, _I, _I, _I], _S),
        "csa_topk_select": ([_I, _I, _L, _I, _I, _I, _P, _I, _P, _P, _S, _P], _I),
        "csa_topk_select_noalloc": ([_I, _I, _L, _I, _I, _I, _P, _P, _P], _I),
        "csa_index_topk_workspace_size": ([_I, _I, _I, _I, _I, _I, _I, _I], _S),
        "csa_index_topk": ([_I, _I, _L, _I, _I, _I, _I, _I, _P, _I, _P, _P, _I, _P, _P, _I, _I, _P, _P, _S, _P], _I),
        "csa_index_topk_varlen": ([_I, _I, _P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _I, _P, _P, _I, _I, _P, _P, _S,
                                   _P], _I),
        "csa_decode_append": ([_I, _I, _I, _I, _L, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _P,
                               _P], _I),
        "csa_sparse_attn_workspace_size": ([_I, _I, _I, _I, _I], _S),
        "csa_sparse_attn": ([_I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _I, _P, _P, _P, _P, _S, _P], _I),
        "hca_attn": ([_I, _I, _L, _I, _I, _I, _I, _I, _F, _P, _P, _P, _I, _P, _P, _P], _I),
        "swa_attn": ([_I, _I, _L, _I, _I, _I, _I, _I, _F, _P, _P, _P, _I, _P, _P, _P], _I),
        "csa_device_status": ([_P], _I),
        "csa_last_error": ([], C.c_char_p),
        "csa_wait_selftest": ([C.c_uint32, _P, _P], _I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(st: int):
    if st != 0:
        raise CsaError(st, load().csa_last_error().decode())


def _arr(ctype, vals):
    return (ctype * len(vals))(*vals)


# ---- the C entry points, same names and argument order ----------------------

def csa_compress(B, n, m, logits, xs, x_dtypes, dims, outs, out_dtypes, out_scales=None, stream=None):
    ns = len(xs)
    xp = _arr(C.c_void_p, [_ptr(x) for x in xs])
    op = _arr(C.c_void_p, [_ptr(o) for o in outs])
    sp = None if out_scales is None else _arr(C.c_void_p, [_ptr(s) for s in out_scales])
    _check(load().csa_compress(B, n, m, _ptr(logits), ns, xp, _arr(C.c_int, x_dtypes), _arr(C.c_int, dims),
                               op, _arr(C.c_int, out_dtypes), sp, _stream(stream)))


def csa_compress_per_channel(B, n, m, logits, xs, x_dtypes, dims, outs, out_dtypes, out_scales=None, stream=None):
    """logits: one [B, n, dim] fp32 tensor per stream."""
    ns = len(xs)
    lp = _arr(C.c_void_p, [_ptr(lg) for lg in logits])
    xp = _arr(C.c_void_p, [_ptr(x) for x in xs])
    op = _arr(C.c_void_p, [_ptr(o) for o in outs])
    sp = None if out_scales is None else _arr(C.c_void_p, [_ptr(s) for s in out_scales])
    _check(load().csa_compress_per_channel(B, n, m, ns, lp, xp, _arr(C.c_int, x_dtypes), _arr(C.c_int, dims), op,
                                           _arr(C.c_int, out_dtypes), sp, _stream(stream)))


def csa_index_scores_workspace_size(B, N_c, d_I, k_dtype):
    return load().csa_index_scores_workspace_size(B, N_c, d_I, k_dtype)


def csa_index_scores(B, n_q, q_pos0, m, N_c, H_I, d_I, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                     scores, workspace=None, workspace_bytes=0, stream=None, head_weight=None, relu=False):
    """scores: an fp32 or bf16 tensor; its dtype is the score_dtype passed on.
    head_weight / relu (keywords) are the C arguments that follow k_scale."""
    _check(load().csa_index_scores(B, n_q, q_pos0, m, N_c, H_I, d_I, _ptr(q_idx), q_dtype, _ptr(q_scale),
                                   _ptr(k_idx), k_dtype, _ptr(k_scale), _ptr(head_weight), 1 if relu else 0,
                                   _ptr(scores), dtype_code(scores.dtype), _ptr(workspace), workspace_bytes,
                                   _stream(stream)))


def csa_topk_select_workspace_size(B, n_q, N_c, k):
    return load().csa_topk_select_workspace_size(B, n_q, N_c, k)


def csa_topk_select(B, n_q, q_pos0, m, N_c, k, scores, topk, workspace=None, workspace_bytes=0, stream=None):
    """scores: an fp32 or bf16 tensor; its dtype is the score_dtype passed on."""
    _check(load().csa_topk_select(B, n_q, q_pos0, m, N_c, k, _ptr(scores), dtype_code(scores.dtype), _ptr(topk),
                                  _ptr(workspace), workspace_bytes, _stream(stream)))


def csa_topk_select_noalloc(B, n_q, q_pos0, m, N_c, k, scores, topk, stream=None):
    """csa_topk_select without a workspace, for callers that cannot allocate
    device memory; the library uses its fixed built-in scratch array instead."""
    _check(load().csa_topk_select_noalloc(B, n_q, q_pos0, m, N_c, k, _ptr(scores), _ptr(topk), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 4 << 20


def csa_index_topk_workspace_size(B, n_q, N_c, H_I, d_I, k, k_dtype, score_dtype=F32):
    return load().csa_index_topk_workspace_size(B, n_q, N_c, H_I, d_I, k, k_dtype, score_dtype)


def csa_index_topk(B, n_q, q_pos0, m, N_c, H_I, d_I, k, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                   topk, workspace, workspace_bytes, stream=None, score_dtype=F32, head_weight=None, relu=False):
    """head_weight, relu and score_dtype (keywords) are the C arguments
    between k_scale and topk."""
    _check(load().csa_index_topk(B, n_q, q_pos0, m, N_c, H_I, d_I, k, _ptr(q_idx), q_dtype, _ptr(q_scale),
                                 _ptr(k_idx), k_dtype, _ptr(k_scale), _ptr(head_weight), 1 if relu else 0,
                                 score_dtype, _ptr(topk), _ptr(workspace), workspace_bytes, _stream(stream)))


def csa_index_topk_varlen(B, n_q, lens, m, N_c, H_I, d_I, k, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                          topk, workspace, workspace_bytes, stream=None, score_dtype=F32, head_weight=None,
                          relu=False):
    """lens: device int64 [B]; keywords as in csa_index_topk."""
    _check(load().csa_index_topk_varlen(B, n_q, _ptr(lens), m, N_c, H_I, d_I, k, _ptr(q_idx), q_dtype,
                                        _ptr(q_scale), _ptr(k_idx), k_dtype, _ptr(k_scale), _ptr(head_weight),
                                        1 if relu else 0, score_dtype, _ptr(topk), _ptr(workspace),
                                        workspace_bytes, _stream(stream)))


def csa_decode_append(B, m, d, d_I, N_cap, logit_new, k_new, v_new, ik_new, x_dtype, stage_logits, stage_k,
                      stage_v, stage_ik, lens, k_c, v_c, kv_dtype, ik_c, ik_dtype, ik_scale=None, stream=None):
    _check(load().csa_decode_append(B, m, d, d_I, N_cap, _ptr(logit_new), _ptr(k_new), _ptr(v_new), _ptr(ik_new),
                                    x_dtype, _ptr(stage_logits), _ptr(stage_k), _ptr(stage_v), _ptr(stage_ik),
                                    _ptr(lens), _ptr(k_c), _ptr(v_c), kv_dtype, _ptr(ik_c), ik_dtype,
                                    _ptr(ik_scale), _stream(stream)))


def csa_sparse_attn_workspace_size(B, n_q, H, d, k):
    return load().csa_sparse_attn_workspace_size(B, n_q, H, d, k)


def csa_sparse_attn(B, n_q, H, d, N_c, k, scale, q, k_c, v_c, dtype, topk, out, lse=None, workspace=None,
                    workspace_bytes=0, stream=None, H_kv=1):
    """H_kv (keyword) is the C argument after H."""
    _check(load().csa_sparse_attn(B, n_q, H, H_kv, d, N_c, k, scale, _ptr(q), _ptr(k_c), _ptr(v_c), dtype,
                                  _ptr(topk), _ptr(out), _ptr(lse), _ptr(workspace), workspace_bytes,
                                  _stream(stream)))


def hca_attn(B, n_q, q_pos0, m, N_c, H, d, scale, q, k_c, v_c, dtype, out, lse=None, stream=None, H_kv=1):
    """H_kv (keyword) is the C argument after H."""
    _check(load().hca_attn(B, n_q, q_pos0, m, N_c, H, H_kv, d, scale, _ptr(q), _ptr(k_c), _ptr(v_c), dtype,
                           _ptr(out), _ptr(lse), _stream(stream)))


def swa_attn(B, n_q, q_pos0, n_kv, window, H, d, scale, q, k, v, dtype, out, lse=None, stream=None, H_kv=1):
    """H_kv (keyword) is the C argument after H."""
    _check(load().swa_attn(B, n_q, q_pos0, n_kv, window, H, H_kv, d, scale, _ptr(q), _ptr(k), _ptr(v), dtype,
                           _ptr(out), _ptr(lse), _stream(stream)))


def csa_device_status(stream=None):
    _check(load().csa_device_status(_stream(stream)))


def csa_last_error() -> str:
    return load().csa_last_error().decode()


def csa_wait_selftest(limit_us, aborted, stream=None):
    _check(load().csa_wait_selftest(limit_us, _ptr(aborted), _stream(stream)))


# ---- conveniences: dtype codes and output allocation (no compute) ---------

def dtype_code(t: torch.dtype) -> int:
    return {torch.float32: F32, torch.bfloat16: BF16}[t]


def empty_workspace(nbytes: int, device="cuda"):
    """Caller-owned workspace buffer (at least 16 bytes, 256-byte aligned by torch)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)
