"""ctypes binding of libmla (include/mla.h): argument marshalling only.

Every function takes CUDA torch tensors, passes their device pointers, sizes
and the current stream to the C entry point of the same name, and raises
``MLAError`` on a non-OK status.  Outputs and workspaces not supplied by the
caller are allocated with torch (the library itself allocates nothing).
There is no CPU path: if the library cannot be loaded, importing a function
raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# MLA_CHECKS=1 in the environment selects the build with the kernels' own
# work-split checks and NaN-filled shared memory (build.py --checks).
CHECKS = os.environ.get("MLA_CHECKS", "0") == "1"
LIB_PATH = os.path.join(HERE, "libmla_checks.so" if CHECKS else "libmla.so")

MLA_BF16, MLA_FP32 = 0, 1
STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
          4: "MLA_ERR_TIMEOUT", 5: "MLA_ERR_DEVICE_BOUNDS"}

SYMBOLS = ["mla_absorb_q", "mla_decode_workspace_size", "mla_decode_attn", "mla_combine_splits",
           "mla_out_proj_workspace_size", "mla_out_proj", "mla_get_device_status",
           "mla_status_string", "mla_version", "mla_set_decode_events", "mla_launch_count",
           "mla_decode_plan", "mla_decode_attn_noalloc", "mla_decode_noalloc_max_bytes",
           "mla_cache_append_workspace_size", "mla_cache_append", "mla_project_q_workspace_size",
           "mla_project_q", "mla_fold_out_weights", "mla_out_proj_merged_workspace_size",
           "mla_out_proj_merged", "mla_set_wait_limit", "mla_decode_attn_partial",
           "mla_prefill_expand", "mla_prefill_attn", "mla_prefill_workspace_size", "mla_prefill_out",
           "mla_fold_q_workspace_size", "mla_fold_q_weights", "mla_absorb_q_merged"]


class MLAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {STATUS.get(code, code)} ({_lib().mla_status_string(code).decode()})")


_LIB = None


def _lib():
    """Load libmla.so (building it in-tree first if it is missing or stale)."""
    global _LIB
    if _LIB is None:
        from . import build
        if build.stale(CHECKS):
            build.build(checks=CHECKS)
        lib = ctypes.CDLL(LIB_PATH)
        P, I, L, F, Z = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                         ctypes.c_size_t)
        lib.mla_absorb_q.argtypes = [P, P, P, I, I, I, I, I, P]
        lib.mla_absorb_q.restype = I
        lib.mla_decode_workspace_size.argtypes = [I, I, I, I, I]
        lib.mla_decode_workspace_size.restype = Z
        lib.mla_decode_attn.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, L, F, I, P, P, P, Z,
                                        I, P]
        lib.mla_decode_attn.restype = I
        lib.mla_combine_splits.argtypes = [P, P, I, L, I, P, P, I, P]
        lib.mla_combine_splits.restype = I
        lib.mla_out_proj_workspace_size.argtypes = [I, I, I, I, I]
        lib.mla_out_proj_workspace_size.restype = Z
        lib.mla_out_proj.argtypes = [P, P, P, P, P, I, I, I, I, I, P, Z, I, P]
        lib.mla_out_proj.restype = I
        lib.mla_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        lib.mla_get_device_status.restype = I
        lib.mla_status_string.argtypes = [I]
        lib.mla_status_string.restype = ctypes.c_char_p
        lib.mla_version.argtypes = []
        lib.mla_version.restype = I
        lib.mla_set_decode_events.argtypes = [P, P]
        lib.mla_set_decode_events.restype = None
        lib.mla_launch_count.argtypes = []
        lib.mla_launch_count.restype = ctypes.c_uint64
        lib.mla_decode_plan.argtypes = [P, I, I, I, I, I, I, P, L]
        lib.mla_decode_plan.restype = L
        lib.mla_decode_attn_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, L, F, I, P,
                                                P, I, P]
        lib.mla_decode_attn_noalloc.restype = I
        lib.mla_decode_noalloc_max_bytes.argtypes = []
        lib.mla_decode_noalloc_max_bytes.restype = Z
        D = ctypes.c_double
        lib.mla_cache_append_workspace_size.argtypes = [I, I, I, I]
        lib.mla_cache_append_workspace_size.restype = Z
        lib.mla_cache_append.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, L, D, P, Z, I, P]
        lib.mla_cache_append.restype = I
        lib.mla_project_q_workspace_size.argtypes = [I, I, I, I, I, I]
        lib.mla_project_q_workspace_size.restype = Z
        lib.mla_project_q.argtypes = [P, P, P, P, P, I, I, I, I, I, D, P, Z, I, P]
        lib.mla_project_q.restype = I
        lib.mla_fold_out_weights.argtypes = [P, P, P, I, I, I, I, I, P]
        lib.mla_fold_out_weights.restype = I
        lib.mla_out_proj_merged_workspace_size.argtypes = [I, I, I, I, I]
        lib.mla_out_proj_merged_workspace_size.restype = Z
        lib.mla_out_proj_merged.argtypes = [P, P, P, I, I, I, I, P, Z, I, P]
        lib.mla_out_proj_merged.restype = I
        lib.mla_decode_attn_partial.argtypes = lib.mla_decode_attn.argtypes
        lib.mla_decode_attn_partial.restype = I
        lib.mla_prefill_expand.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P]
        lib.mla_prefill_expand.restype = I
        lib.mla_prefill_attn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, I, P]
        lib.mla_prefill_attn.restype = I
        lib.mla_prefill_workspace_size.argtypes = [I, I, I, I, I]
        lib.mla_prefill_workspace_size.restype = Z
        lib.mla_prefill_out.argtypes = [P, P, P, I, I, I, I, P, Z, I, P]
        lib.mla_prefill_out.restype = I
        lib.mla_fold_q_workspace_size.argtypes = [I, I, I, I]
        lib.mla_fold_q_workspace_size.restype = Z
        lib.mla_fold_q_weights.argtypes = [P, P, P, I, I, I, I, I, P, Z, I, P]
        lib.mla_fold_q_weights.restype = I
        lib.mla_absorb_q_merged.argtypes = [P, P, P, I, I, I, I, I, P]
        lib.mla_absorb_q_merged.restype = I
        lib.mla_set_wait_limit.argtypes = [ctypes.c_uint64]
        lib.mla_set_wait_limit.restype = I
        _LIB = lib
    return _LIB


def library():
    """The loaded ctypes library handle."""
    return _lib()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MLA_BF16
    if t.dtype == torch.float32:
        return MLA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmla takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libmla takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        raise MLAError(fn, code)


# ------------------------------------------------------------------- entries

def absorb_q(q_nope: torch.Tensor, w_uk: torch.Tensor, q_lat: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """q_lat[r,i,:] = W^UK_i^T q_nope[r,i,:]; q_nope [rows,H,d_h], w_uk [H,d_h,d_c]."""
    rows, H, d_h = q_nope.shape
    d_c = w_uk.shape[2]
    if q_lat is None:
        q_lat = torch.empty((rows, H, d_c), dtype=q_nope.dtype, device=q_nope.device)
    _check("mla_absorb_q", _lib().mla_absorb_q(_ptr(q_nope), _ptr(w_uk), _ptr(q_lat), rows, H, d_h,
                                               d_c, _dt(q_nope), _stream(stream)))
    return q_lat


def decode_workspace_size(B: int, T: int, H: int, d_c: int, dtype=torch.bfloat16) -> int:
    return int(_lib().mla_decode_workspace_size(B, T, H, d_c,
                                                MLA_BF16 if dtype == torch.bfloat16 else MLA_FP32))


def decode_attn(q_lat, q_pe, kv_pool, page_table, seq_lens, scale: float, causal: bool = False,
                o=None, lse=None, workspace=None, seq_lens_host=None, stream=None):
    """Paged absorbed decode; returns (o [B,T,H,d_c], lse [B,T,H] fp32)."""
    B, T, H, d_c = q_lat.shape
    d_r = q_pe.shape[3]
    num_pages, page, width = kv_pool.shape
    max_pages = page_table.shape[1]
    if o is None:
        o = torch.empty_like(q_lat)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q_lat.device)
    dt = _dt(q_lat)
    need = int(_lib().mla_decode_workspace_size(B, T, H, d_c, dt))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_lat.device)
    host = None
    if seq_lens_host is not None:
        seq_lens_host = seq_lens_host.to(torch.int32).contiguous()
        host = ctypes.c_void_p(seq_lens_host.data_ptr())
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("mla_decode_attn", _lib().mla_decode_attn(
        _ptr(q_lat), _ptr(q_pe), _ptr(kv_pool), _ptr(page_table), _ptr(seq_lens), host, B, T, H,
        d_c, d_r, page, max_pages, num_pages, float(scale), int(bool(causal)), _ptr(o), _ptr(lse),
        _ptr(workspace), ws_bytes, dt, _stream(stream)))
    return o, lse


def decode_attn_partial(q_lat, q_pe, kv_pool, page_table, seq_lens, scale: float,
                        causal: bool = False, o=None, lse=None, workspace=None,
                        seq_lens_host=None, stream=None):
    """decode_attn with o in fp32 (a part's normalised result, for merging
    with other parts by combine_splits); returns (o fp32, lse)."""
    B, T, H, d_c = q_lat.shape
    d_r = q_pe.shape[3]
    num_pages, page, width = kv_pool.shape
    max_pages = page_table.shape[1]
    if o is None:
        o = torch.empty((B, T, H, d_c), dtype=torch.float32, device=q_lat.device)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q_lat.device)
    if o.dtype != torch.float32:
        raise TypeError("decode_attn_partial writes an fp32 o")
    dt = _dt(q_lat)
    need = int(_lib().mla_decode_workspace_size(B, T, H, d_c, dt))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_lat.device)
    host = None
    if seq_lens_host is not None:
        seq_lens_host = seq_lens_host.to(torch.int32).contiguous()
        host = ctypes.c_void_p(seq_lens_host.data_ptr())
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("mla_decode_attn_partial", _lib().mla_decode_attn_partial(
        _ptr(q_lat), _ptr(q_pe), _ptr(kv_pool), _ptr(page_table), _ptr(seq_lens), host, B, T, H,
        d_c, d_r, page, max_pages, num_pages, float(scale), int(bool(causal)), _ptr(o), _ptr(lse),
        _ptr(workspace), ws_bytes, dt, _stream(stream)))
    return o, lse


def decode_attn_noalloc(q_lat, q_pe, kv_pool, page_table, seq_lens, scale: float,
                        causal: bool = False, o=None, lse=None, seq_lens_host=None, stream=None):
    """decode_attn through mla_decode_attn_noalloc: the same result, with the
    library's fixed internal scratch instead of a caller workspace (for
    callers that cannot allocate device memory; the caller still provides
    inputs and outputs).  Returns (o, lse)."""
    B, T, H, d_c = q_lat.shape
    d_r = q_pe.shape[3]
    num_pages, page, width = kv_pool.shape
    max_pages = page_table.shape[1]
    if o is None:
        o = torch.empty_like(q_lat)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q_lat.device)
    host = None
    if seq_lens_host is not None:
        seq_lens_host = seq_lens_host.to(torch.int32).contiguous()
        host = ctypes.c_void_p(seq_lens_host.data_ptr())
    _check("mla_decode_attn_noalloc", _lib().mla_decode_attn_noalloc(
        _ptr(q_lat), _ptr(q_pe), _ptr(kv_pool), _ptr(page_table), _ptr(seq_lens), host, B, T, H,
        d_c, d_r, page, max_pages, num_pages, float(scale), int(bool(causal)), _ptr(o), _ptr(lse),
        _dt(q_lat), _stream(stream)))
    return o, lse


def noalloc_max_bytes() -> int:
    """Size of the fixed scratch array behind decode_attn_noalloc."""
    return int(_lib().mla_decode_noalloc_max_bytes())


def combine_splits(o_part, lse_part, o=None, lse=None, out_dtype=torch.bfloat16, stream=None):
    """Merge [S, rows, d_c] fp32 partials and their [S, rows] lse; returns (o, lse)."""
    S, rows, d_c = o_part.shape
    if o is None:
        o = torch.empty((rows, d_c), dtype=out_dtype, device=o_part.device)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=o_part.device)
    _check("mla_combine_splits", _lib().mla_combine_splits(
        _ptr(o_part), _ptr(lse_part), S, rows, d_c, _ptr(o), _ptr(lse), _dt(o), _stream(stream)))
    return o, lse


def out_proj_workspace_size(rows: int, H: int, d_h: int, d: int, dtype=torch.bfloat16) -> int:
    return int(_lib().mla_out_proj_workspace_size(
        rows, H, d_h, d, MLA_BF16 if dtype == torch.bfloat16 else MLA_FP32))


def out_proj(o, w_uv, w_o, v_tmp=None, out=None, workspace=None, stream=None):
    """out = W^O concat_i(W^UV_i o_i); o [rows,H,d_c], w_uv [H,d_h,d_c], w_o [d,H*d_h]."""
    rows, H, d_c = o.shape
    d_h = w_uv.shape[1]
    d = w_o.shape[0]
    if v_tmp is None:
        v_tmp = torch.empty((rows, H * d_h), dtype=o.dtype, device=o.device)
    if out is None:
        out = torch.empty((rows, d), dtype=o.dtype, device=o.device)
    need = out_proj_workspace_size(rows, H, d_h, d, o.dtype)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=o.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("mla_out_proj", _lib().mla_out_proj(
        _ptr(o), _ptr(w_uv), _ptr(w_o), _ptr(v_tmp), _ptr(out), rows, H, d_h, d_c, d,
        _ptr(workspace), ws_bytes, _dt(o), _stream(stream)))
    return out


def fold_out_weights(w_uv, w_o, w_merged=None, stream=None):
    """W_merged [d, H*d_c] with row n, head slice i = W^UV_i^T W^O[n, i*d_h:(i+1)*d_h]."""
    H, d_h, d_c = w_uv.shape
    d = w_o.shape[0]
    if w_merged is None:
        w_merged = torch.empty((d, H * d_c), dtype=w_uv.dtype, device=w_uv.device)
    _check("mla_fold_out_weights", _lib().mla_fold_out_weights(
        _ptr(w_uv), _ptr(w_o), _ptr(w_merged), H, d_h, d_c, d, _dt(w_uv), _stream(stream)))
    return w_merged


def out_proj_merged(o, w_merged, out=None, workspace=None, stream=None):
    """out = W_merged concat_i o_i; o [rows,H,d_c], w_merged [d,H*d_c]."""
    rows, H, d_c = o.shape
    d = w_merged.shape[0]
    if out is None:
        out = torch.empty((rows, d), dtype=o.dtype, device=o.device)
    need = int(_lib().mla_out_proj_merged_workspace_size(rows, H, d_c, d, _dt(o)))
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=o.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("mla_out_proj_merged", _lib().mla_out_proj_merged(
        _ptr(o), _ptr(w_merged), _ptr(out), rows, H, d_c, d, _ptr(workspace), ws_bytes, _dt(o),
        _stream(stream)))
    return out


def cache_append_workspace_size(N: int, d: int, d_c: int, dtype=torch.bfloat16) -> int:
    return int(_lib().mla_cache_append_workspace_size(
        N, d, d_c, MLA_BF16 if dtype == torch.bfloat16 else MLA_FP32))


def cache_append(h, w_dkv, w_kr, seq_ids, positions, page_table, kv_pool,
                 rope_base: float = 10000.0, workspace=None, stream=None):
    """Write [W^DKV h_n ; RoPE(W^KR h_n, pos_n)] for each token n into its pool row.

    h [N,d], w_dkv [d_c,d], w_kr [d_r,d], seq_ids / positions [N] int32,
    page_table [B,max_pages] int32, kv_pool [num_pages,page,d_c+d_r]
    (updated in place).  Returns kv_pool.
    """
    N, d = h.shape
    d_c, d_r = w_dkv.shape[0], w_kr.shape[0]
    B, max_pages = page_table.shape
    num_pages, page, _ = kv_pool.shape
    need = cache_append_workspace_size(N, d, d_c, h.dtype)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=h.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("mla_cache_append", _lib().mla_cache_append(
        _ptr(h), _ptr(w_dkv), _ptr(w_kr), _ptr(seq_ids), _ptr(positions), _ptr(page_table),
        _ptr(kv_pool), N, d, d_c, d_r, B, page, max_pages, num_pages, float(rope_base),
        _ptr(workspace), ws_bytes, _dt(h), _stream(stream)))
    return kv_pool


def project_q_workspace_size(N: int, H: int, d_h: int, d_r: int, d: int,
                             dtype=torch.bfloat16) -> int:
    return int(_lib().mla_project_q_workspace_size(
        N, H, d_h, d_r, d, MLA_BF16 if dtype == torch.bfloat16 else MLA_FP32))


def project_q(h, w_q, positions, H: int, d_h: int, d_r: int, q_nope=None, q_pe=None,
              rope_base: float = 10000.0, workspace=None, stream=None):
    """q = W^Q h per head [q^C ; q^R], q^R rotated at each token's position.

    h [N,d], w_q [H*(d_h+d_r),d], positions [N] int32.  Returns
    (q_nope [N,H,d_h], q_pe [N,H,d_r]).
    """
    N, d = h.shape
    if q_nope is None:
        q_nope = torch.empty((N, H, d_h), dtype=h.dtype, device=h.device)
    if q_pe is None:
        q_pe = torch.empty((N, H, d_r), dtype=h.dtype, device=h.device)
    need = project_q_workspace_size(N, H, d_h, d_r, d, h.dtype)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=h.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("mla_project_q", _lib().mla_project_q(
        _ptr(h), _ptr(w_q), _ptr(positions), _ptr(q_nope), _ptr(q_pe), N, H, d_h, d_r, d,
        float(rope_base), _ptr(workspace), ws_bytes, _dt(h), _stream(stream)))
    return q_nope, q_pe


def get_device_status(stream=None) -> tuple[int, int]:
    """(status code, detail) of the current device; reads and clears the word."""
    detail = ctypes.c_uint32(0)
    code = _lib().mla_get_device_status(_stream(stream), ctypes.byref(detail))
    return int(code), int(detail.value)


def fold_q_weights(w_uk, w_q, d_r: int, w_merged=None, workspace=None, stream=None):
    """W_merged [d_q, H, d_c] with [k, i, :] = W^UK_i^T W^UQ_i[:, k]; w_uk
    [H, d_h, d_c], w_q [H*(d_h+d_r), d_q]."""
    H, d_h, d_c = w_uk.shape
    d_q = w_q.shape[1]
    if w_merged is None:
        w_merged = torch.empty((d_q, H, d_c), dtype=w_uk.dtype, device=w_uk.device)
    need = int(_lib().mla_fold_q_workspace_size(H, d_h, d_q, _dt(w_uk)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=w_uk.device)
    _check("mla_fold_q_weights", _lib().mla_fold_q_weights(
        _ptr(w_uk), _ptr(w_q), _ptr(w_merged), H, d_h, d_r, d_c, d_q, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _dt(w_uk), _stream(stream)))
    return w_merged


def absorb_q_merged(c_q, w_merged, q_lat=None, stream=None):
    """q_lat [rows, H, d_c] = W_merged c^Q; c_q [rows, d_q], w_merged [d_q, H, d_c]."""
    rows, d_q = c_q.shape
    _, H, d_c = w_merged.shape
    if q_lat is None:
        q_lat = torch.empty((rows, H, d_c), dtype=c_q.dtype, device=c_q.device)
    _check("mla_absorb_q_merged", _lib().mla_absorb_q_merged(
        _ptr(c_q), _ptr(w_merged), _ptr(q_lat), rows, H, d_c, d_q, _dt(c_q), _stream(stream)))
    return q_lat


def prefill_expand(kv, w_uk, w_uv, k_nope=None, v=None, stream=None):
    """Per-head keys and values of cache rows kv [rows, d_c+d_r]:
    (k_nope, v) [rows, H, d_h] = (W^UK_i c, W^UV_i c)."""
    rows, width = kv.shape
    H, d_h, d_c = w_uk.shape
    if k_nope is None:
        k_nope = torch.empty((rows, H, d_h), dtype=kv.dtype, device=kv.device)
    if v is None:
        v = torch.empty((rows, H, d_h), dtype=kv.dtype, device=kv.device)
    _check("mla_prefill_expand", _lib().mla_prefill_expand(
        _ptr(kv), _ptr(w_uk), _ptr(w_uv), _ptr(k_nope), _ptr(v), rows, H, d_h, d_c, width - d_c,
        _dt(kv), _stream(stream)))
    return k_nope, v


def prefill_attn(q_nope, q_pe, k_nope, kv, v, L: int, scale: float, causal: bool = True, u=None,
                 lse=None, stream=None):
    """Attention of B = rows / L sequences, every token a query; q_nope, k_nope,
    v [rows, H, d_h], q_pe [rows, H, d_r], kv [rows, d_c+d_r].  Returns
    (u [rows, H, d_h], lse [rows, H] fp32)."""
    rows, H, d_h = q_nope.shape
    d_r = q_pe.shape[2]
    d_c = kv.shape[1] - d_r
    if rows % L:
        raise ValueError("rows must be a multiple of L")
    if u is None:
        u = torch.empty_like(q_nope)
    if lse is None:
        lse = torch.empty((rows, H), dtype=torch.float32, device=q_nope.device)
    _check("mla_prefill_attn", _lib().mla_prefill_attn(
        _ptr(q_nope), _ptr(q_pe), _ptr(k_nope), _ptr(kv), _ptr(v), rows // L, L, H, d_h, d_c, d_r,
        float(scale), int(bool(causal)), _ptr(u), _ptr(lse), _dt(q_nope), _stream(stream)))
    return u, lse


def prefill_out(u, w_o, out=None, workspace=None, stream=None):
    """out [rows, d] = W^O u for u [rows, H, d_h], w_o [d, H*d_h]."""
    rows, H, d_h = u.shape
    d = w_o.shape[0]
    if out is None:
        out = torch.empty((rows, d), dtype=u.dtype, device=u.device)
    need = int(_lib().mla_prefill_workspace_size(rows, H, d_h, d, _dt(u)))
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=u.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("mla_prefill_out", _lib().mla_prefill_out(
        _ptr(u), _ptr(w_o), _ptr(out), rows, H, d_h, d, _ptr(workspace), ws_bytes, _dt(u),
        _stream(stream)))
    return out


def set_wait_limit(ns: int) -> None:
    """How long the library's kernels wait for a pipeline step before giving
    up with MLA_ERR_TIMEOUT (ns; 0 restores the default of 2 s)."""
    _check("mla_set_wait_limit", _lib().mla_set_wait_limit(int(ns)))


def set_decode_events(start: torch.cuda.Event | None, end: torch.cuda.Event | None) -> None:
    """Record `start`/`end` around the attention kernel of later bf16 decode calls."""
    if start is None or end is None:
        _lib().mla_set_decode_events(None, None)
    else:
        _lib().mla_set_decode_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(end.cuda_event))


def launch_count() -> int:
    """Kernels this library has launched in this process."""
    return int(_lib().mla_launch_count())


def decode_plan(seq_lens, T: int, H: int, max_pages: int, causal: bool = False,
                clusters: int = 0):
    """Pieces of the bf16 decode work split (host computation), as a list of
    dicts with keys cluster, unit, lp0, lp1, slot, g_first, g_last."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    B = lens.shape[0]
    lib = _lib()
    n = lib.mla_decode_plan(lens.ctypes.data_as(ctypes.c_void_p), B, T, H, max_pages,
                            int(bool(causal)), clusters, None, 0)
    if n < 0:
        raise ValueError("mla_decode_plan: bad arguments")
    out = np.zeros((max(n, 1), 7), dtype=np.int64)
    lib.mla_decode_plan(lens.ctypes.data_as(ctypes.c_void_p), B, T, H, max_pages,
                        int(bool(causal)), clusters, out.ctypes.data_as(ctypes.c_void_p), n)
    keys = ["cluster", "unit", "lp0", "lp1", "slot", "g_first", "g_last"]
    return [dict(zip(keys, map(int, row))) for row in out[:n]]
