"""Python binding of lcattn: CSA + HCA compressed attention on one B300.

Thin ctypes layer over ``liblcattn.so`` (built from ``csrc/`` for sm_103a).
Every function has the name of the C entry point it calls and only marshals
arguments: torch tensors provide device memory and the current CUDA stream;
all arithmetic runs in the library's CUDA kernels.  There is no CPU fallback:
if the library is missing or no CUDA device is present, calls raise.

Shapes and meanings are those of ``include/lcattn.h``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblcattn.so")

LC_OK, LC_ERR_INVALID_ARG, LC_ERR_UNSUPPORTED, LC_ERR_CUDA, LC_ERR_TIMEOUT = 0, 1, 2, 3, 4
LC_ERR_DEVICE_CHECK, LC_ERR_WORKSPACE = 5, 6
LC_F32, LC_BF16 = 0, 1
LC_DEVERR_INDEX, LC_DEVERR_WINDOW, LC_DEVERR_BATCH, LC_DEVERR_TIMEOUT = 1, 2, 4, 8
LC_DEVERR_SINK = 16
LC_OP_LIGHTNING_INDEX, LC_OP_TOPK_SELECT, LC_OP_SPARSE_MQA_ATTN, LC_OP_HCA_DENSE_ATTN = 0, 1, 2, 3

ENTRY_POINTS = ("csa_compress", "hca_compress", "token_gated_compress", "rope_rotate",
                "decode_append", "lightning_index", "topk_select", "mx_quantize",
                "lightning_index_mx",
                "sparse_mqa_attn", "hca_dense_attn", "lc_workspace_size", "lc_status_string",
                "lc_last_cuda_error", "lc_launch_count", "lc_last_kernel", "lc_version",
                "lc_debug_stall")
LC_STALL_INDEX_TC, LC_STALL_SPARSE_TC, LC_STALL_HCA_TC = 1, 2, 4


class LCError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class _LcBatch(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("cu_q", ctypes.c_void_p), ("q_pos0", ctypes.c_void_p),
                ("cu_c", ctypes.c_void_p), ("cu_raw", ctypes.c_void_p),
                ("raw_pos0", ctypes.c_void_p), ("total_q", ctypes.c_int64),
                ("max_q", ctypes.c_int64), ("max_c", ctypes.c_int64),
                ("total_c", ctypes.c_int64), ("total_raw", ctypes.c_int64)]


class _LcDecodeLayer(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("R", ctypes.c_int32), ("d", ctypes.c_int32),
                ("m", ctypes.c_int32), ("HI", ctypes.c_int32), ("dI", ctypes.c_int32),
                ("cap", ctypes.c_int64), ("n_tok", ctypes.c_void_p),
                ("Kring", ctypes.c_void_p), ("Vring", ctypes.c_void_p),
                ("kI_ring", ctypes.c_void_p), ("Kc", ctypes.c_void_p), ("Vc", ctypes.c_void_p),
                ("kI", ctypes.c_void_p), ("q_pos0", ctypes.c_void_p), ("cu_raw", ctypes.c_void_p),
                ("raw_pos0", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblcattn.so (no CUDA device needed to load it)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"liblcattn.so not built at {path}; run "
                          "`python -m long_context_compressed_13_b300._build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
    bp = ctypes.POINTER(_LcBatch)
    sig = {
        "csa_compress": [vp, vp, vp, vp, i64, i32, i32, i32, vp, vp, i64, vp],
        "hca_compress": [vp, vp, vp, vp, i64, i32, i32, i32, vp, vp, i64, vp],
        "token_gated_compress": [vp, vp, i64, i32, i32, i32, vp, i64, vp],
        "rope_rotate": [vp, i64, i32, i32, i64, i32, i32, vp],
        "lightning_index": [vp, vp, vp, bp, i32, i32, i32, i32, vp, i64, i32, vp, vp, sz, vp, vp],
        "topk_select": [vp, i64, bp, i32, i32, vp, vp, sz, vp, vp],
        "mx_quantize": [vp, i64, i32, i32, vp, vp, vp],
        "lightning_index_mx": [i32, vp, vp, vp, vp, vp, bp, i32, i32, i32, vp, i64, i32, vp, vp,
                               sz, vp, vp],
        "sparse_mqa_attn": [vp, vp, vp, vp, i32, vp, vp, bp, i32, i32, i32, i32, f32, vp, i32, i32,
                            vp, vp, vp, sz, vp, vp],
        "hca_dense_attn": [vp, vp, vp, vp, vp, bp, i32, i32, i32, i32, f32, vp, i32, i32, vp, vp,
                           vp, sz, vp, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i32
    lib.decode_append.argtypes = [ctypes.POINTER(_LcDecodeLayer), vp, vp, vp, vp, vp, vp, i32, vp,
                                  vp]
    lib.decode_append.restype = i32
    lib.lc_workspace_size.argtypes = [i32, bp, i32, i32, i32, i32, i32]
    lib.lc_workspace_size.restype = sz
    lib.lc_status_string.argtypes = [i32]
    lib.lc_status_string.restype = ctypes.c_char_p
    lib.lc_last_cuda_error.restype = i32
    lib.lc_launch_count.restype = ctypes.c_uint64
    lib.lc_last_kernel.restype = ctypes.c_char_p
    lib.lc_debug_stall.argtypes = [ctypes.c_uint32, ctypes.c_int64]
    lib.lc_debug_stall.restype = None
    lib.lc_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def launch_count() -> int:
    """Kernels the library has enqueued in this process."""
    return int(load_library().lc_launch_count())


def last_kernel() -> str:
    """Name of the last kernel the library launched from this thread."""
    return load_library().lc_last_kernel().decode()


def debug_stall(kernels: int, clocks: int) -> None:
    """Test hook: the named tensor-core kernels (LC_STALL_* mask) start with a
    bounded wait of `clocks` SM clocks on a barrier nothing completes, so
    their waits run out; clocks <= 0 turns it off."""
    load_library().lc_debug_stall(kernels, clocks)


def _check(fn: str, status: int):
    if status != LC_OK:
        lib = load_library()
        msg = lib.lc_status_string(status).decode()
        if status == LC_ERR_CUDA:
            msg += (f" (cudaError {lib.lc_last_cuda_error()}; last kernel launched: "
                    f"{lib.lc_last_kernel().decode() or 'none'})")
        raise LCError(fn, status, msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LC_F32
    if t.dtype == torch.bfloat16:
        return LC_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(t: Optional[torch.Tensor], name: str, dtype=None) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


@dataclass
class DeviceBatch:
    """lc_batch with its arrays on the device.  Build with from_host()."""
    B: int
    cu_q: torch.Tensor
    q_pos0: torch.Tensor
    cu_c: torch.Tensor
    cu_raw: torch.Tensor
    raw_pos0: torch.Tensor
    total_q: int
    max_q: int
    max_c: int
    total_c: int = 0
    total_raw: int = 0
    host: object = None

    @staticmethod
    def from_host(cu_q: Sequence[int], q_pos0: Sequence[int], cu_c: Sequence[int],
                  cu_raw: Sequence[int], raw_pos0: Sequence[int], device="cuda") -> "DeviceBatch":
        B = len(q_pos0)
        if not (len(cu_q) == len(cu_c) == len(cu_raw) == B + 1 and len(raw_pos0) == B):
            raise ValueError("batch arrays have inconsistent lengths")
        mk = lambda a: torch.tensor(list(a), dtype=torch.int64, device=device)
        nq = [cu_q[b + 1] - cu_q[b] for b in range(B)]
        nc = [cu_c[b + 1] - cu_c[b] for b in range(B)]
        return DeviceBatch(B, mk(cu_q), mk(q_pos0), mk(cu_c), mk(cu_raw), mk(raw_pos0),
                           int(cu_q[-1]), max(nq) if nq else 0, max(nc) if nc else 0,
                           int(cu_c[-1]), int(cu_raw[-1]))

    @staticmethod
    def from_workload(batch, device="cuda") -> "DeviceBatch":
        db = DeviceBatch.from_host(batch.cu_q, batch.q_pos0, batch.cu_c, batch.cu_raw,
                                   batch.raw_pos0, device=device)
        db.host = batch
        return db

    def c_struct(self) -> _LcBatch:
        return _LcBatch(self.B, self.cu_q.data_ptr(), self.q_pos0.data_ptr(),
                        self.cu_c.data_ptr(), self.cu_raw.data_ptr(), self.raw_pos0.data_ptr(),
                        self.total_q, self.max_q, self.max_c, self.total_c, self.total_raw)


def workspace_size(op: int, batch: DeviceBatch, H=0, d=0, HI=0, dI=0, k=0) -> int:
    cb = batch.c_struct()
    return int(load_library().lc_workspace_size(op, ctypes.byref(cb), H, d, HI, dI, k))


def _rope_pos0(rope_pos0) -> int:
    if rope_pos0 is None:
        return -1
    if rope_pos0 < 0:
        raise ValueError("rope_pos0 is a position (>= 0) or None")
    return int(rope_pos0)


def _compress(fn_name, K, V, G_K, G_V, m, Kc=None, Vc=None, stream=None, rope_pos0=None):
    lib = load_library()
    T, d = K.shape
    if V.shape != K.shape or V.dtype != K.dtype:
        raise ValueError("K and V must have the same shape and dtype")
    if Kc is None:
        Kc = torch.empty((T // m, d), dtype=K.dtype, device=K.device)
    if Vc is None:
        Vc = torch.empty((T // m, d), dtype=K.dtype, device=K.device)
    if Kc.shape[0] < T // m or Vc.shape[0] < T // m:
        raise ValueError("output too small")
    st = getattr(lib, fn_name)(_dev(K, "K"), _dev(V, "V"), _dev(G_K, "G_K", torch.float32),
                               _dev(G_V, "G_V", torch.float32), T, d, m, _dtype_code(K),
                               _dev(Kc, "Kc", K.dtype), _dev(Vc, "Vc", K.dtype),
                               _rope_pos0(rope_pos0), _stream(stream))
    _check(fn_name, st)
    return Kc, Vc


def csa_compress(K, V, G_K, G_V=None, m: int = 4, Kc=None, Vc=None, stream=None,
                 rope_pos0=None):
    """K, V [T,d] -> (Kc, Vc) [floor(T/m), d]; gates [m,d] fp32.  rope_pos0:
    position of K[0] to give every entry partial RoPE at its last token, or
    None."""
    return _compress("csa_compress", K, V, G_K, G_K if G_V is None else G_V, m, Kc, Vc, stream,
                     rope_pos0)


def hca_compress(K, V, G_K, G_V=None, m: int = 128, Kc=None, Vc=None, stream=None,
                 rope_pos0=None):
    """K, V [T,d] -> (Kc, Vc) [floor(T/m), d]; gates [m,d] fp32 (rope_pos0 as
    for csa_compress)."""
    return _compress("hca_compress", K, V, G_K, G_K if G_V is None else G_V, m, Kc, Vc, stream,
                     rope_pos0)


def rope_rotate(X, pos0: int, inverse: bool = False, stream=None):
    """Partial RoPE, in place, of rows X[i] ([n, d] or [n, heads, d]) at
    positions pos0 + i (inverse: rotate back).  Returns X."""
    lib = load_library()
    n, d = X.shape[0], X.shape[-1]
    hv = int(np.prod(X.shape[1:-1])) if X.dim() > 2 else 1
    st = lib.rope_rotate(_dev(X, "X"), n, hv, d, int(pos0), 1 if inverse else 0, _dtype_code(X),
                         _stream(stream))
    _check("rope_rotate", st)
    return X


def token_gated_compress(X, Z, m: int, Xc=None, stream=None, rope_pos0=None):
    """X [T, d] with per-token gate logits Z [T, d] fp32 -> Xc [floor(T/m), d].
    X may also be [T, H_I, d_I] (token-level indexer keys); Xc then has the
    same trailing shape."""
    lib = load_library()
    T = X.shape[0]
    d = int(np.prod(X.shape[1:]))
    if tuple(Z.shape) != tuple(X.shape):
        raise ValueError("Z must hold one fp32 gate logit per element of X (same shape)")
    if Xc is None:
        Xc = torch.empty((T // m, *X.shape[1:]), dtype=X.dtype, device=X.device)
    if Xc.shape[0] < T // m:
        raise ValueError("output too small")
    st = lib.token_gated_compress(_dev(X, "X"), _dev(Z, "Z", torch.float32), T, d, m,
                                  _dtype_code(X), _dev(Xc, "Xc", X.dtype), _rope_pos0(rope_pos0),
                                  _stream(stream))
    _check("token_gated_compress", st)
    return Xc


def lightning_index(qI, w, kI, batch: DeviceBatch, m: int, *, scores: bool | torch.Tensor = True,
                    k: int = 0, topk: bool | torch.Tensor = False, ws=None, dev_err=None,
                    stream=None):
    """Indexer scores [total_q, max_c] (fp32, -inf where invisible) and/or
    the fused top-k [total_q, k].  Returns (scores or None, topk or None)."""
    lib = load_library()
    Nq, HI, dI = qI.shape
    if isinstance(scores, torch.Tensor):
        sc = scores
    elif scores:
        sc = torch.empty((Nq, max(batch.max_c, 1)), dtype=torch.float32, device=qI.device)
    else:
        sc = None
    if isinstance(topk, torch.Tensor):
        tk = topk
    elif topk:
        tk = torch.empty((Nq, k), dtype=torch.int32, device=qI.device)
    else:
        tk = None
    if tk is not None and sc is None and ws is None:
        need = workspace_size(LC_OP_LIGHTNING_INDEX, batch, HI=HI, dI=dI, k=k)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=qI.device)
    cb = batch.c_struct()
    ld = sc.shape[1] if sc is not None else 0
    st = lib.lightning_index(_dev(qI, "qI"), _dev(w, "w", torch.float32), _dev(kI, "kI", qI.dtype),
                             ctypes.byref(cb), HI, dI, m, _dtype_code(qI), _dev(sc, "scores"),
                             ld, k, _dev(tk, "topk", torch.int32), _dev(ws, "ws"),
                             ws.numel() if ws is not None else 0,
                             _dev(dev_err, "dev_err", torch.int32), _stream(stream))
    _check("lightning_index", st)
    return sc, tk


LC_MXFP8, LC_MXFP4 = 8, 4  # OCP MX element formats E4M3 and E2M1


def mx_quantize(X, fmt: int, codes=None, scales=None, stream=None):
    """MX quantization (blocks of 32 consecutive values, one E8M0 scale each).
    X [..., D] fp32/bf16, D % 32 == 0 -> (codes uint8 [..., D] for MXFP8 or
    [..., D/2] for MXFP4 (even value in the low nibble), scales uint8
    [..., D/32])."""
    lib = load_library()
    D = X.shape[-1]
    if D % 32:
        raise ValueError(f"the last dimension ({D}) must be a multiple of 32")
    lead = tuple(X.shape[:-1])
    if codes is None:
        codes = torch.empty(lead + (D if fmt == LC_MXFP8 else D // 2,), dtype=torch.uint8,
                            device=X.device)
    if scales is None:
        scales = torch.empty(lead + (D // 32,), dtype=torch.uint8, device=X.device)
    st = lib.mx_quantize(_dev(X, "X"), X.numel(), fmt, _dtype_code(X),
                         _dev(codes, "codes", torch.uint8), _dev(scales, "scales", torch.uint8),
                         _stream(stream))
    _check("mx_quantize", st)
    return codes, scales


def lightning_index_mx(fmt: int, qc, qs, w, kc, ks, batch: DeviceBatch, m: int, *,
                       scores: bool | torch.Tensor = True, k: int = 0,
                       topk: bool | torch.Tensor = False, ws=None, dev_err=None, stream=None):
    """The indexer on MX-quantized q_I (qc [Nq, HI, dI*bits/8], qs [Nq, HI, dI/32])
    and k_I (kc, ks likewise over the entries), as returned by mx_quantize.
    Returns (scores or None, topk or None) like lightning_index."""
    lib = load_library()
    Nq, HI = qc.shape[0], qc.shape[1]
    dI = qc.shape[2] * 8 // fmt
    if isinstance(scores, torch.Tensor):
        sc = scores
    elif scores:
        sc = torch.empty((Nq, max(batch.max_c, 1)), dtype=torch.float32, device=qc.device)
    else:
        sc = None
    if isinstance(topk, torch.Tensor):
        tk = topk
    elif topk:
        tk = torch.empty((Nq, k), dtype=torch.int32, device=qc.device)
    else:
        tk = None
    if tk is not None and sc is None and ws is None:
        need = workspace_size(LC_OP_LIGHTNING_INDEX, batch, HI=HI, dI=dI, k=k)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=qc.device)
    cb = batch.c_struct()
    ld = sc.shape[1] if sc is not None else 0
    st = lib.lightning_index_mx(fmt, _dev(qc, "qc", torch.uint8), _dev(qs, "qs", torch.uint8),
                                _dev(w, "w", torch.float32), _dev(kc, "kc", torch.uint8),
                                _dev(ks, "ks", torch.uint8), ctypes.byref(cb), HI, dI, m,
                                _dev(sc, "scores"), ld, k, _dev(tk, "topk", torch.int32),
                                _dev(ws, "ws"), ws.numel() if ws is not None else 0,
                                _dev(dev_err, "dev_err", torch.int32), _stream(stream))
    _check("lightning_index_mx", st)
    return sc, tk


def topk_select(scores, batch: DeviceBatch, m: int, k: int, topk=None, dev_err=None,
                stream=None):
    """scores [total_q, ld] fp32 -> topk [total_q, k] int32."""
    lib = load_library()
    if topk is None:
        topk = torch.empty((scores.shape[0], k), dtype=torch.int32, device=scores.device)
    cb = batch.c_struct()
    st = lib.topk_select(_dev(scores, "scores", torch.float32), scores.shape[1], ctypes.byref(cb),
                         m, k, _dev(topk, "topk", torch.int32), None, 0,
                         _dev(dev_err, "dev_err", torch.int32), _stream(stream))
    _check("topk_select", st)
    return topk


def _sink_ptr(sink, Q) -> int:
    """Device pointer of the per-head sink logits [H] fp32 (0 for none)."""
    if sink is None:
        return 0
    H = Q.shape[1]
    if sink.numel() != H:
        raise ValueError(f"sink must hold one fp32 logit per head ({H}), got {sink.numel()}")
    if sink.device != Q.device:
        raise ValueError(f"sink is on {sink.device}, Q on {Q.device}")
    return _dev(sink, "sink", torch.float32)


def sparse_mqa_attn(Q, Kc, Vc, topk, Kraw, Vraw, batch: DeviceBatch, m: int, W: int,
                    scale: float, O=None, lse: bool | torch.Tensor = True, dev_err=None,
                    stream=None, sink=None, rope: bool = False):
    """CSA core attention.  Returns (O [total_q,H,d], lse [total_q,H] or None).
    sink: per-head attention-sink logits [H] fp32 on the device, or None.
    rope: partial RoPE (Q rotated at t, O rotated back; Kc/Vc and the raw
    window must hold rotated entries and tokens)."""
    lib = load_library()
    Nq, H, d = Q.shape
    if O is None:
        O = torch.empty_like(Q)
    if isinstance(lse, torch.Tensor):
        L = lse
    elif lse:
        L = torch.empty((Nq, H), dtype=torch.float32, device=Q.device)
    else:
        L = None
    cb = batch.c_struct()
    st = lib.sparse_mqa_attn(_dev(Q, "Q"), _dev(Kc, "Kc", Q.dtype), _dev(Vc, "Vc", Q.dtype),
                             _dev(topk, "topk", torch.int32), topk.shape[1],
                             _dev(Kraw, "Kraw", Q.dtype), _dev(Vraw, "Vraw", Q.dtype),
                             ctypes.byref(cb), H, d, m, W, float(scale),
                             _sink_ptr(sink, Q), 1 if rope else 0, _dtype_code(Q),
                             _dev(O, "O", Q.dtype), _dev(L, "lse", torch.float32), None, 0,
                             _dev(dev_err, "dev_err", torch.int32), _stream(stream))
    _check("sparse_mqa_attn", st)
    return O, L


def hca_dense_attn(Q, Kc, Vc, Kraw, Vraw, batch: DeviceBatch, m: int, W: int, scale: float,
                   O=None, lse: bool | torch.Tensor = True, dev_err=None, ws=None, stream=None,
                   sink=None, rope: bool = False):
    """HCA dense attention.  Returns (O [total_q,H,d], lse [total_q,H] or None).
    sink and rope: as for sparse_mqa_attn."""
    lib = load_library()
    Nq, H, d = Q.shape
    if O is None:
        O = torch.empty_like(Q)
    if isinstance(lse, torch.Tensor):
        L = lse
    elif lse:
        L = torch.empty((Nq, H), dtype=torch.float32, device=Q.device)
    else:
        L = None
    cb = batch.c_struct()
    st = lib.hca_dense_attn(_dev(Q, "Q"), _dev(Kc, "Kc", Q.dtype), _dev(Vc, "Vc", Q.dtype),
                            _dev(Kraw, "Kraw", Q.dtype), _dev(Vraw, "Vraw", Q.dtype),
                            ctypes.byref(cb), H, d, m, W, float(scale),
                            _sink_ptr(sink, Q), 1 if rope else 0, _dtype_code(Q),
                            _dev(O, "O", Q.dtype), _dev(L, "lse", torch.float32),
                            _dev(ws, "ws"), ws.numel() if ws is not None else 0,
                            _dev(dev_err, "dev_err", torch.int32), _stream(stream))
    _check("hca_dense_attn", st)
    return O, L


class DecodeLayer:
    """Incremental decode state of one layer for B requests (see
    lc_decode_layer in lcattn.h): the classical cache (cap entries a request),
    the mirrored ring of the last R raw tokens, for a CSA layer (HI > 0) the
    indexer keys and the open block's token-level indexer keys, and the batch
    arrays that decode_append advances.  Torch provides the memory; `batch`
    is the descriptor the step's index and attention calls take."""

    def __init__(self, B: int, R: int, d: int, m: int, cap: int, HI: int = 0, dI: int = 0,
                 dtype=torch.bfloat16, device="cuda"):
        z = lambda *shape, dt=dtype: torch.zeros(shape, dtype=dt, device=device)
        self.B, self.R, self.d, self.m, self.cap, self.HI, self.dI = B, R, d, m, cap, HI, dI
        self.dtype = dtype
        self.n_tok = z(B, dt=torch.int64)
        self.Kring, self.Vring = z(B * 2 * R, d), z(B * 2 * R, d)
        self.kI_ring = z(B * m, HI, dI) if HI else None
        self.Kc, self.Vc = z(B * cap, d), z(B * cap, d)
        self.kI = z(B * cap, HI, dI) if HI else None
        self.q_pos0 = z(B, dt=torch.int64)
        self.cu_raw = torch.arange(B + 1, dtype=torch.int64, device=device) * 2 * R
        self.raw_pos0 = z(B, dt=torch.int64)
        cu_q = torch.arange(B + 1, dtype=torch.int64, device=device)
        cu_c = cu_q * cap
        self.batch = DeviceBatch(B, cu_q, self.q_pos0, cu_c, self.cu_raw, self.raw_pos0,
                                 total_q=B, max_q=1, max_c=cap, total_c=B * cap,
                                 total_raw=B * 2 * R)

    def c_struct(self) -> _LcDecodeLayer:
        p = lambda t: t.data_ptr() if t is not None else 0
        return _LcDecodeLayer(self.B, self.R, self.d, self.m, self.HI, self.dI, self.cap,
                              p(self.n_tok), p(self.Kring), p(self.Vring), p(self.kI_ring),
                              p(self.Kc), p(self.Vc), p(self.kI), p(self.q_pos0),
                              p(self.cu_raw), p(self.raw_pos0))


def decode_append(layer: DecodeLayer, K_new, V_new, G_K, G_V=None, kI_new=None, G_I=None,
                  dev_err=None, stream=None):
    """Appends one token per request (K_new, V_new [B, d]; kI_new [B, HI, dI]
    for a CSA layer): ring, block entries when a block closes, batch arrays."""
    lib = load_library()
    G_V = G_K if G_V is None else G_V
    cs = layer.c_struct()
    st = lib.decode_append(ctypes.byref(cs), _dev(K_new, "K_new", layer.dtype),
                           _dev(V_new, "V_new", layer.dtype),
                           _dev(kI_new, "kI_new", layer.dtype),
                           _dev(G_K, "G_K", torch.float32), _dev(G_V, "G_V", torch.float32),
                           _dev(G_I, "G_I", torch.float32), _dtype_code(K_new),
                           _dev(dev_err, "dev_err", torch.int32), _stream(stream))
    _check("decode_append", st)
