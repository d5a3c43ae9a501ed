"""fp64 CPU oracle for weight-absorbed MLA decode (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its binding in ``mla_latent_kv_71_b300``) never does, and the two share
no code: the oracle is ``mla_oracle.c`` compiled with gcc, wrapped here with
ctypes.

Every function takes numpy arrays.  Floating-point inputs may be float64,
float32, or bf16 bit patterns stored as uint16 (see ``bf16_bits``); the C code
widens each element exactly to double and never rounds an intermediate.

Parity status of each function (what pins it is listed in the tests):
  cache_numbers, score_cost ... pinned to the printed page values
  rope ........................ pinned by closed forms and invariants
  absorb_q, out_proj .......... pinned by the naive-vs-absorbed identity
  decode_attn ................. pinned by a library routine (SDPA), closed
                                forms, invariants and the naive route
  combine ..................... pinned by the split identity
  weight_spread ............... (test infrastructure: the sensitivity of o
                                to rounding the weights, used by the parity
                                bar) pinned by closed forms and by perturbing
                                the weights
  project, naive_decode ....... pinned by a library routine (SDPA) and the
                                identity against the absorbed route
  naive_prefill ............... pinned by naive_decode with T = L and by a
                                library routine (causal SDPA)
  prefill_attn ................ pinned by naive_prefill on exact expansions
                                and by a library routine (causal SDPA)
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library (gcc, OpenMP)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", *extra_flags,
           src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; returns the CDLL."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_D = ctypes.c_double


def _declare(lib):
    lib.orc_cache_numbers.argtypes = [_L, _L, _L, _L, _L, _P]
    lib.orc_score_cost.argtypes = [_L, _L, _L, _P]
    lib.orc_rope.argtypes = [_P, _I, _D, _D]
    lib.orc_absorb_q.argtypes = [_P, _I, _P, _I, _I, _I, _I, _I, _P]
    lib.orc_decode_attn.argtypes = [_P, _I, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                    _I, _I, _D, _I, _P, _L, _P, _P]
    lib.orc_naive_prefill.argtypes = [_P, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _I,
                                      _I, _D, _I, _P, _L, _P, _P]
    lib.orc_prefill_attn.argtypes = [_P, _I, _P, _I, _P, _I, _P, _I, _L, _L, _P, _I, _I, _I, _I,
                                     _I, _I, _D, _I, _P, _L, _P, _P]
    lib.orc_weight_spread.argtypes = [_P, _I, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                      _I, _I, _D, _I, _P, _L, _P]
    lib.orc_attention_weights.argtypes = [_P, _I, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I,
                                          _I, _I, _D, _I, _I, _I, _I, _P]
    lib.orc_attention_weights.restype = _L
    lib.orc_combine.argtypes = [_P, _I, _P, _I, _I, _L, _I, _P, _P]
    lib.orc_out_proj.argtypes = [_P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P]
    lib.orc_project.argtypes = [_P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I,
                                _I, _I, _D, _P, _P, _P]
    lib.orc_naive_decode.argtypes = [_P, _P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I,
                                     _I, _I, _I, _I, _I, _I, _D, _I, _P, _P]
    return lib


def bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor -> its bit patterns as a uint16 numpy array."""
    import torch
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _arr(x):
    """(contiguous array, dtype tag) for a float64/float32/bf16-bits array or torch tensor."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.bfloat16:
                return bf16_bits(x), BF16
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


def _i32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ wrappers

def cache_numbers(h, d_h, h_kv, d_c, d_r, lib=None):
    """Cached numbers per token per layer: dict MHA/GQA/MQA/MLA_latent/MLA."""
    lib = lib or load()
    out = np.zeros(5, dtype=np.int64)
    lib.orc_cache_numbers(h, d_h, h_kv, d_c, d_r, _ptr(out))
    return dict(zip(["MHA", "GQA", "MQA", "MLA_latent", "MLA"], out.tolist()))


def score_cost(n, hd, d_c, lib=None):
    """(key-side, query-side) multiply-add counts for n cached tokens."""
    lib = lib or load()
    out = np.zeros(2, dtype=np.int64)
    lib.orc_score_cost(n, hd, d_c, _ptr(out))
    return int(out[0]), int(out[1])


def rope(x, pos, base=10000.0, lib=None):
    """RoPE of one vector at position pos (returns a new float64 array)."""
    lib = lib or load()
    y = np.array(x, dtype=np.float64, copy=True)
    lib.orc_rope(_ptr(y), y.shape[0], float(pos), float(base))
    return y


def absorb_q(q_nope, w_uk, lib=None):
    """q_nope [R,H,d_h], w_uk [H,d_h,d_c] -> q_lat [R,H,d_c] float64."""
    lib = lib or load()
    q, dq = _arr(q_nope)
    w, dw = _arr(w_uk)
    R, H, d_h = q.shape
    d_c = w.shape[2]
    out = np.empty((R, H, d_c), dtype=np.float64)
    lib.orc_absorb_q(_ptr(q), dq, _ptr(w), dw, R, H, d_h, d_c, _ptr(out))
    return out


def decode_attn(q_lat, q_pe, pool, page_table, seq_lens, scale, causal=False, sel=None,
                lib=None):
    """Paged absorbed decode.

    q_lat [B,T,H,d_c], q_pe [B,T,H,d_r], pool [P,page,d_c+d_r],
    page_table [B,max_pages] int32, seq_lens [B] int32.
    Returns (o [B,T,H,d_c], lse [B,T,H]) float64, or, with sel (flattened
    (b*T+t)*H+i indices), (o [n,d_c], lse [n]) for those rows only.
    """
    lib = lib or load()
    ql, dql = _arr(q_lat)
    qp, dqp = _arr(q_pe)
    pl, dp = _arr(pool)
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    B, T, H, d_c = ql.shape
    d_r = qp.shape[3]
    page = pl.shape[1]
    max_pages = pt.shape[1]
    assert pl.shape[2] == d_c + d_r
    if sel is None:
        n = B * T * H
        sel_arr = None
    else:
        sel_arr = np.ascontiguousarray(sel, dtype=np.int64)
        n = sel_arr.shape[0]
    o = np.empty((n, d_c), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    lib.orc_decode_attn(_ptr(ql), dql, _ptr(qp), dqp, _ptr(pl), dp, _ptr(pt), _ptr(sl),
                        B, T, H, d_c, d_r, page, max_pages, float(scale), int(bool(causal)),
                        _ptr(sel_arr) if sel_arr is not None else None, n, _ptr(o), _ptr(lse))
    if sel is None:
        return o.reshape(B, T, H, d_c), lse.reshape(B, T, H)
    return o, lse


def weight_spread(q_lat, q_pe, pool, page_table, seq_lens, scale, causal=False, sel=None,
                  lib=None):
    """D[.., c] = sum_j a_j |c_j[c] - o[c]| for every (b, t, i), or for the
    flattened indices in sel: how far o can move when the weights a_j are
    perturbed by relative errors of at most u (by u / (1 - u) * D).  Not a
    step of the method: the parity bar uses it to bound what rounding the
    softmax weights to bf16 can do.  Shapes as decode_attn's o."""
    lib = lib or load()
    ql, dql = _arr(q_lat)
    qp, dqp = _arr(q_pe)
    pl, dp = _arr(pool)
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    B, T, H, d_c = ql.shape
    d_r = qp.shape[3]
    if sel is None:
        n, sel_arr = B * T * H, None
    else:
        sel_arr = np.ascontiguousarray(sel, dtype=np.int64)
        n = sel_arr.shape[0]
    D = np.empty((n, d_c), dtype=np.float64)
    lib.orc_weight_spread(_ptr(ql), dql, _ptr(qp), dqp, _ptr(pl), dp, _ptr(pt), _ptr(sl), B, T, H,
                          d_c, d_r, pl.shape[1], pt.shape[1], float(scale), int(bool(causal)),
                          _ptr(sel_arr) if sel_arr is not None else None, n, _ptr(D))
    return D.reshape(B, T, H, d_c) if sel is None else D


def attention_weights(q_lat, q_pe, pool, page_table, seq_lens, scale, b, t, i,
                      causal=False, lib=None):
    """Softmax row a_j of one (b, t, i) as a float64 array."""
    lib = lib or load()
    ql, dql = _arr(q_lat)
    qp, dqp = _arr(q_pe)
    pl, dp = _arr(pool)
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    B, T, H, d_c = ql.shape
    d_r = qp.shape[3]
    a = np.empty((max(int(sl[b]), 1),), dtype=np.float64)
    n = lib.orc_attention_weights(_ptr(ql), dql, _ptr(qp), dqp, _ptr(pl), dp, _ptr(pt),
                                  _ptr(sl), T, H, d_c, d_r, pl.shape[1], pt.shape[1],
                                  float(scale), int(bool(causal)), b, t, i, _ptr(a))
    return a[:n]


def combine(o_part, lse_part, lib=None):
    """o_part [S,N,d_c], lse_part [S,N] -> (o [N,d_c], lse [N]) float64."""
    lib = lib or load()
    op, dpo = _arr(o_part)
    lp, dpl = _arr(lse_part)
    S, N, d_c = op.shape
    o = np.empty((N, d_c), dtype=np.float64)
    lse = np.empty((N,), dtype=np.float64)
    lib.orc_combine(_ptr(op), dpo, _ptr(lp), dpl, S, N, d_c, _ptr(o), _ptr(lse))
    return o, lse


def out_proj(o, w_uv, w_o, lib=None):
    """o [R,H,d_c], w_uv [H,d_h,d_c], w_o [d,H*d_h] -> (out [R,d], u [R,H*d_h])."""
    lib = lib or load()
    oo, dov = _arr(o)
    wu, dwu = _arr(w_uv)
    wo, dwo = _arr(w_o)
    R, H, d_c = oo.shape
    d_h = wu.shape[1]
    d = wo.shape[0]
    out = np.empty((R, d), dtype=np.float64)
    u = np.empty((R, H * d_h), dtype=np.float64)
    lib.orc_out_proj(_ptr(oo), dov, _ptr(wu), dwu, _ptr(wo), dwo, R, H, d_h, d_c, d,
                     _ptr(out), _ptr(u))
    return out, u


def project(h, w_dkv, w_kr, w_q, H, d_h, qpos, rope_base=10000.0, lib=None):
    """Hidden states -> (cache [B*L, d_c+d_r], q_nope [B,H,d_h], q_pe [B,H,d_r])."""
    lib = lib or load()
    hh, dht = _arr(h)
    w1, dw1 = _arr(w_dkv)
    w2, dw2 = _arr(w_kr)
    w3, dw3 = _arr(w_q)
    B, L, d = hh.shape
    d_c = w1.shape[0]
    d_r = w2.shape[0]
    cache = np.empty((B * L, d_c + d_r), dtype=np.float64)
    q_nope = np.empty((B, H, d_h), dtype=np.float64)
    q_pe = np.empty((B, H, d_r), dtype=np.float64)
    lib.orc_project(_ptr(hh), dht, _ptr(w1), dw1, _ptr(w2), dw2, _ptr(w3), dw3, B, L, d, H,
                    d_h, d_c, d_r, int(qpos), float(rope_base), _ptr(cache), _ptr(q_nope),
                    _ptr(q_pe))
    return cache, q_nope, q_pe


def naive_decode(cache, q_nope, q_pe, w_uk, w_uv, w_o, L, scale, causal=False, lib=None):
    """Naive (expand K and V) decode on a contiguous cache [B*L, d_c+d_r].

    q_nope [B,T,H,d_h], q_pe [B,T,H,d_r], w_uk/w_uv [H,d_h,d_c], w_o [d,H*d_h]
    (w_o may be None).  Returns (u [B,T,H,d_h], out [B,T,d] or None).
    """
    lib = lib or load()
    cc = np.ascontiguousarray(cache, dtype=np.float64)
    qn, dqn = _arr(q_nope)
    qp, dqp = _arr(q_pe)
    wk, dwk = _arr(w_uk)
    wv, dwv = _arr(w_uv)
    B, T, H, d_h = qn.shape
    d_r = qp.shape[3]
    d_c = wk.shape[2]
    u = np.empty((B, T, H, d_h), dtype=np.float64)
    if w_o is not None:
        wo, dwo = _arr(w_o)
        d = wo.shape[0]
        out = np.empty((B, T, d), dtype=np.float64)
        wo_p, out_p = _ptr(wo), _ptr(out)
    else:
        dwo, d, out, wo_p, out_p = F64, 0, None, None, None
    lib.orc_naive_decode(_ptr(cc), _ptr(qn), dqn, _ptr(qp), dqp, _ptr(wk), dwk, _ptr(wv),
                         dwv, wo_p, dwo, B, T, L, H, d_h, d_c, d_r, d, float(scale),
                         int(bool(causal)), _ptr(u), out_p)
    return u, out


def naive_prefill(cache, q_nope, q_pe, w_uk, w_uv, scale, causal=True, sel=None, lib=None):
    """Training-form attention with every token a query.

    cache [B, L, d_c+d_r] rows [c ; k^R]; q_nope [B,L,H,d_h], q_pe [B,L,H,d_r];
    w_uk / w_uv [H,d_h,d_c].  Returns (u [B,L,H,d_h], lse [B,L,H]) float64, or
    with sel (flattened (b*L + t)*H + i rows) (u [n,d_h], lse [n]).
    """
    lib = lib or load()
    cc = np.ascontiguousarray(cache, dtype=np.float64)
    B, L = cc.shape[0], cc.shape[1]
    cc = cc.reshape(B * L, -1)
    qn, dqn = _arr(q_nope)
    qp, dqp = _arr(q_pe)
    wk, dwk = _arr(w_uk)
    wv, dwv = _arr(w_uv)
    H, d_h = qn.shape[2], qn.shape[3]
    d_r = qp.shape[3]
    d_c = wk.shape[2]
    if sel is None:
        n, sel_arr = B * L * H, None
    else:
        sel_arr = np.ascontiguousarray(sel, dtype=np.int64)
        n = sel_arr.shape[0]
    u = np.empty((n, d_h), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    lib.orc_naive_prefill(_ptr(cc), _ptr(qn), dqn, _ptr(qp), dqp, _ptr(wk), dwk, _ptr(wv), dwv,
                          B, L, H, d_h, d_c, d_r, float(scale), int(bool(causal)),
                          _ptr(sel_arr) if sel_arr is not None else None, n, _ptr(u), _ptr(lse))
    if sel is None:
        return u.reshape(B, L, H, d_h), lse.reshape(B, L, H)
    return u, lse


def prefill_attn(q_nope, q_pe, k_nope, k_pe, v, L, scale, causal=True, k_pe_off=0, sel=None,
                 lib=None):
    """Attention of given per-head keys and values, every token a query.

    q_nope, k_nope, v [rows, H, d_h]; q_pe [rows, H, d_r]; k_pe [rows, w] with
    the RoPE key in columns k_pe_off .. k_pe_off + d_r - 1 (cache rows work
    as they are); rows = B * L.  Returns (u [rows, H, d_h], lse [rows, H])
    float64, or with sel (flattened token * H + head rows) (u [n, d_h], lse [n]).
    """
    lib = lib or load()
    qn, dqn = _arr(q_nope)
    qp, dqp = _arr(q_pe)
    kn, dkn = _arr(k_nope)
    kp, dkp = _arr(k_pe)
    vv, dv = _arr(v)
    rows, H, d_h = qn.shape
    d_r = qp.shape[2]
    B = rows // L
    if sel is None:
        n, sel_arr = rows * H, None
    else:
        sel_arr = np.ascontiguousarray(sel, dtype=np.int64)
        n = sel_arr.shape[0]
    u = np.empty((n, d_h), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    lib.orc_prefill_attn(_ptr(qn), dqn, _ptr(qp), dqp, _ptr(kn), dkn, _ptr(kp), dkp, kp.shape[1],
                         int(k_pe_off), _ptr(vv), dv, B, L, H, d_h, d_r, float(scale),
                         int(bool(causal)), _ptr(sel_arr) if sel_arr is not None else None, n,
                         _ptr(u), _ptr(lse))
    if sel is None:
        return u.reshape(rows, H, d_h), lse.reshape(rows, H)
    return u, lse
