"""Plain fp64 CPU oracle for the CSA + HCA attention path.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may call it; the library's product path never does.  It shares no
code with the CUDA library.  The arithmetic lives in ``oracle.c`` (plain C,
fp64, OpenMP over query rows); this module only builds it with gcc and
marshals numpy arrays.

Each wrapper works on ONE sequence; ragged batches loop over sequences here.
The function-level citations are in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            D = ctypes.POINTER(ctypes.c_double)
            I64 = ctypes.POINTER(ctypes.c_int64)
            I32 = ctypes.POINTER(ctypes.c_int32)
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_compress.argtypes = [D, D, i64, i32, i32, D]
            lib.oracle_compress.restype = None
            lib.oracle_compress_tok.argtypes = [D, D, i64, i32, i32, D]
            lib.oracle_compress_tok.restype = None
            lib.oracle_rope.argtypes = [D, I64, i64, i32, i32, i32, dbl, i32, D]
            lib.oracle_rope.restype = None
            U32 = ctypes.POINTER(ctypes.c_uint32)
            U8 = ctypes.POINTER(ctypes.c_uint8)
            lib.oracle_mx_quantize.argtypes = [D, i64, i32, U32, U8, D]
            lib.oracle_mx_quantize.restype = None
            lib.oracle_index.argtypes = [D, D, D, I64, i64, i64, i32, i32, i32, D]
            lib.oracle_index.restype = None
            lib.oracle_topk.argtypes = [D, i64, i64, I64, i32, I32]
            lib.oracle_topk.restype = None
            lib.oracle_sparse_attn.argtypes = [D, D, D, i64, I32, i32, D, D, i64, i64,
                                               I64, i64, i32, i32, i32, dbl, D, D, D]
            lib.oracle_sparse_attn.restype = i64
            lib.oracle_hca_attn.argtypes = [D, D, D, i64, i32, D, D, i64, i64,
                                            I64, i64, i32, i32, i32, dbl, D, D, D]
            lib.oracle_hca_attn.restype = i64
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def n_visible(t, m: int):
    """Entries visible from absolute position t: floor((t+1)/m)."""
    return (np.asarray(t, dtype=np.int64) + 1) // m


def compress(X, G, m: int) -> np.ndarray:
    """X [T, d], G [m, d] -> Xc [floor(T/m), d] (fp64)."""
    X, G = _f64(X), _f64(G)
    T, d = X.shape
    assert G.shape == (m, d)
    out = np.zeros((T // m, d), dtype=np.float64)
    _load().oracle_compress(_p(X, ctypes.c_double), _p(G, ctypes.c_double), T, d, m,
                            _p(out, ctypes.c_double))
    return out


def compress_tok(X, Z, m: int) -> np.ndarray:
    """Token-gated compressor: X [T, d], per-token gate logits Z [T, d] ->
    Xc [floor(T/m), d] (fp64)."""
    X, Z = _f64(X), _f64(Z)
    T, d = X.shape
    assert Z.shape == (T, d)
    out = np.zeros((T // m, d), dtype=np.float64)
    _load().oracle_compress_tok(_p(X, ctypes.c_double), _p(Z, ctypes.c_double), T, d, m,
                                _p(out, ctypes.c_double))
    return out


ROPE_DIMS = 64
ROPE_BASE = 10000.0


def rope(X, pos, inverse: bool = False) -> np.ndarray:
    """Partial RoPE of the last 64 dimensions.  X [n, d] or [n, H, d], pos [n]
    (every vector of row r at position pos[r]); inverse rotates by -pos."""
    X, pos = _f64(X), _i64(pos)
    shape = X.shape
    n, d = shape[0], shape[-1]
    hd = int(np.prod(shape[1:-1])) if len(shape) > 2 else 1
    assert pos.shape == (n,) and d >= ROPE_DIMS
    Y = np.zeros_like(X)
    _load().oracle_rope(_p(X, ctypes.c_double), _p(pos, ctypes.c_int64), n, hd, d, ROPE_DIMS,
                        ROPE_BASE, -1 if inverse else 1, _p(Y, ctypes.c_double))
    return Y


def entry_positions(pos0: int, n: int, m: int) -> np.ndarray:
    """Position of each compressed entry: its last token, pos0 + (j+1) m - 1."""
    return pos0 + (np.arange(n, dtype=np.int64) + 1) * m - 1


MXFP8, MXFP4 = 8, 4  # element formats E4M3 and E2M1 (OCP MX v1.0)
MX_BLOCK = 32


def mx_quantize(X, fmt: int):
    """MX quantization of X (its size a multiple of 32; blocks of 32
    consecutive values in row-major order).  Returns (codes, scales, deq):
    per value its element bit pattern (uint8; E2M1 codes are 4-bit), per
    block the E8M0 scale byte, and the dequantized values (fp64, X's shape)."""
    X = _f64(X)
    n = X.size
    assert n % MX_BLOCK == 0 and fmt in (MXFP8, MXFP4)
    codes = np.zeros(n, dtype=np.uint32)
    scales = np.zeros(n // MX_BLOCK, dtype=np.uint8)
    deq = np.zeros(n, dtype=np.float64)
    _load().oracle_mx_quantize(_p(X.reshape(-1), ctypes.c_double), n, fmt,
                               _p(codes, ctypes.c_uint32), _p(scales, ctypes.c_uint8),
                               _p(deq, ctypes.c_double))
    return codes.astype(np.uint8).reshape(X.shape), scales, deq.reshape(X.shape)


def index_mx(qI, w, kI, tpos, m: int, fmt: int) -> np.ndarray:
    """The low-precision indexer: q_I and k_I are MX-quantized (blocks of 32
    along each head's d_I values) and the score is the indexer's formula on
    the dequantized values, I[t,j] = sum_h w[t,h] max(0, q^_h . k^_h)."""
    _, _, qd = mx_quantize(qI, fmt)
    _, _, kd = mx_quantize(kI, fmt)
    return index(qd, w, kd, tpos, m)


def index(qI, w, kI, tpos, m: int) -> np.ndarray:
    """qI [Nq, HI, dI], w [Nq, HI], kI [Tc, HI, dI], tpos [Nq] -> I [Nq, Tc]
    (invisible entries = -inf)."""
    qI, w, kI, tpos = _f64(qI), _f64(w), _f64(kI), _i64(tpos)
    Nq, HI, dI = qI.shape
    Tc = kI.shape[0]
    assert kI.shape[1:] == (HI, dI) and w.shape == (Nq, HI) and tpos.shape == (Nq,)
    assert np.all(n_visible(tpos, m) <= Tc), "query sees entries that are not stored"
    out = np.zeros((Nq, Tc), dtype=np.float64)
    _load().oracle_index(_p(qI, ctypes.c_double), _p(w, ctypes.c_double), _p(kI, ctypes.c_double),
                         _p(tpos, ctypes.c_int64), Nq, Tc, HI, dI, m, _p(out, ctypes.c_double))
    return out


def topk(I, nvis, k: int) -> np.ndarray:
    """I [Nq, ld] scores (only columns < nvis[r] are read), nvis [Nq] -> idx [Nq, k] int32."""
    I, nvis = _f64(I), _i64(nvis)
    Nq, ld = I.shape
    assert nvis.shape == (Nq,) and np.all(nvis <= ld) and np.all(nvis >= 0)
    out = np.zeros((Nq, k), dtype=np.int32)
    _load().oracle_topk(_p(I, ctypes.c_double), Nq, ld, _p(nvis, ctypes.c_int64), k,
                        _p(out, ctypes.c_int32))
    return out


def _sink(sink, H):
    """Per-head sink logits as an fp64 pointer, or NULL for none."""
    if sink is None:
        return None, ctypes.cast(None, ctypes.POINTER(ctypes.c_double))
    s = _f64(sink).reshape(-1)
    assert s.shape == (H,)
    # a sink logit is a real number or -inf (no sink for that head)
    if np.any(np.isnan(s) | (s == np.inf)):
        raise ValueError("sink logits must be finite or -inf")
    return s, _p(s, ctypes.c_double)


def sparse_attn(Q, Kc, Vc, idx, Kraw, Vraw, raw_pos0: int, tpos, W: int, scale: float,
                sink=None):
    """CSA core attention for one sequence.  Returns (O [Nq,H,d], lse [Nq,H]).
    sink: per-head sink logits [H] (natural-log units, like scale * q.k) or
    None."""
    Q, Kc, Vc, Kraw, Vraw = _f64(Q), _f64(Kc), _f64(Vc), _f64(Kraw), _f64(Vraw)
    idx, tpos = _i32(idx), _i64(tpos)
    Nq, H, d = Q.shape
    k = idx.shape[1]
    O = np.zeros((Nq, H, d), dtype=np.float64)
    lse = np.zeros((Nq, H), dtype=np.float64)
    keep, sp = _sink(sink, H)
    rc = _load().oracle_sparse_attn(
        _p(Q, ctypes.c_double), _p(Kc, ctypes.c_double), _p(Vc, ctypes.c_double), Kc.shape[0],
        _p(idx, ctypes.c_int32), k, _p(Kraw, ctypes.c_double), _p(Vraw, ctypes.c_double),
        Kraw.shape[0], raw_pos0, _p(tpos, ctypes.c_int64), Nq, H, d, W, scale, sp,
        _p(O, ctypes.c_double), _p(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_sparse_attn: invalid input at row {-rc - 1}")
    return O, lse


def _as_operand(X, operand_dtype):
    """The rotated operand as the method stores it: exact (None) or rounded to
    bf16 (round to nearest even) in the bf16 setting."""
    if operand_dtype is None:
        return X
    import torch
    assert operand_dtype == "bf16"
    return torch.from_numpy(np.ascontiguousarray(X)).to(torch.bfloat16).double().numpy()


def sparse_attn_rope(Q, Kc, Vc, idx, Kraw, Vraw, raw_pos0: int, tpos, W: int, scale: float,
                     m: int, sink=None, operand_dtype=None):
    """CSA attention with partial RoPE, from unrotated inputs, in the order the
    reading fixes: each compressed entry rotated at the position of its last
    token ((j+1) m - 1), each window token at its own position, each query at
    t; attention; the output rotated back at t.  operand_dtype "bf16": the
    rotated q, k and v are bf16 values (the operands of the bf16 setting).
    Returns (O, lse)."""
    Kc, Vc, Kraw, Vraw = _f64(Kc), _f64(Vc), _f64(Kraw), _f64(Vraw)
    ep = entry_positions(0, Kc.shape[0], m)
    rp = raw_pos0 + np.arange(Kraw.shape[0], dtype=np.int64)
    op = lambda X, pos: _as_operand(rope(X, pos), operand_dtype)
    O, lse = sparse_attn(op(Q, tpos), op(Kc, ep), op(Vc, ep), idx, op(Kraw, rp), op(Vraw, rp),
                         raw_pos0, tpos, W, scale, sink)
    return rope(O, tpos, inverse=True), lse


def hca_attn_rope(Q, Kc, Vc, m: int, Kraw, Vraw, raw_pos0: int, tpos, W: int, scale: float,
                  sink=None, operand_dtype=None):
    """HCA attention with partial RoPE, as sparse_attn_rope."""
    Kc, Vc, Kraw, Vraw = _f64(Kc), _f64(Vc), _f64(Kraw), _f64(Vraw)
    ep = entry_positions(0, Kc.shape[0], m)
    rp = raw_pos0 + np.arange(Kraw.shape[0], dtype=np.int64)
    op = lambda X, pos: _as_operand(rope(X, pos), operand_dtype)
    O, lse = hca_attn(op(Q, tpos), op(Kc, ep), op(Vc, ep), m, op(Kraw, rp), op(Vraw, rp),
                      raw_pos0, tpos, W, scale, sink)
    return rope(O, tpos, inverse=True), lse


def hca_attn(Q, Kc, Vc, m: int, Kraw, Vraw, raw_pos0: int, tpos, W: int, scale: float,
             sink=None):
    """HCA attention for one sequence.  Returns (O [Nq,H,d], lse [Nq,H]).
    sink: as for sparse_attn."""
    Q, Kc, Vc, Kraw, Vraw = _f64(Q), _f64(Kc), _f64(Vc), _f64(Kraw), _f64(Vraw)
    tpos = _i64(tpos)
    Nq, H, d = Q.shape
    O = np.zeros((Nq, H, d), dtype=np.float64)
    lse = np.zeros((Nq, H), dtype=np.float64)
    keep, sp = _sink(sink, H)
    rc = _load().oracle_hca_attn(
        _p(Q, ctypes.c_double), _p(Kc, ctypes.c_double), _p(Vc, ctypes.c_double), Kc.shape[0], m,
        _p(Kraw, ctypes.c_double), _p(Vraw, ctypes.c_double), Kraw.shape[0], raw_pos0,
        _p(tpos, ctypes.c_int64), Nq, H, d, W, scale, sp, _p(O, ctypes.c_double),
        _p(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_hca_attn: invalid input at row {-rc - 1}")
    return O, lse
