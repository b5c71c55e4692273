"""Thin ctypes binding of libdspark (include/dspark.h).

Argument marshalling only: every function checks tensor placement, allocates outputs and
workspaces with PyTorch (device memory and streams), and calls the C entry point of the same
name. Nothing here computes any part of the method. A missing library raises: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

c_i32, c_i64, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

DSPARK_BF16, DSPARK_F32 = 0, 1
DSPARK_MAXSUM, DSPARK_WALK, DSPARK_SAMPLE = 0, 1, 2
OP_TOPK, OP_LATTICE, OP_CHAIN, OP_SAMPLE, OP_DENSE_WALK, OP_VERIFY, OP_D2T_CHECK, OP_LATTICE_ROW = range(8)
STATUS = {0: "DSPARK_OK", 1: "DSPARK_EINVAL", 2: "DSPARK_ERANGE", 3: "DSPARK_EDUP", 4: "DSPARK_EPROPOSAL",
          5: "DSPARK_ENONFINITE", 6: "DSPARK_ETIMEOUT", 7: "DSPARK_ECUDA", 8: "DSPARK_EWORKSPACE"}
MODES = {"maxsum": DSPARK_MAXSUM, "walk": DSPARK_WALK, "sample": DSPARK_SAMPLE}

# (name, restype, argtypes) of every symbol include/dspark.h declares
SIGNATURES = [
    ("dspark_workspace_size", c_sz, [c_i32, c_i64, c_i32, c_i64, c_i32]),
    ("dspark_status_string", ctypes.c_char_p, [c_i32]),
    ("dspark_d2t_check", c_i32, [c_vp, c_i64, c_i64, c_i32, c_vp, c_sz, c_vp, c_vp]),
    ("dspark_d2t_check_noalloc", c_i32, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp]),
    ("dspark_topk", c_i32, [c_vp, c_i32, c_i64, c_i32, c_i64, c_i64, c_vp, c_i32, c_f32, c_f32, c_vp, c_i64,
                            c_vp, c_vp, c_vp, c_vp, c_vp]),
    ("dspark_lattice_score", c_i32, [c_vp, c_vp, c_i64, c_i32, c_i32, c_vp, c_vp, c_i32, c_i64, c_i32, c_vp, c_vp,
                                     c_i32, c_i32, c_i64, c_vp, c_vp, c_vp, c_vp, c_vp]),
    ("dspark_lattice_chain", c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_vp, c_vp, c_i32, c_i64, c_i32, c_vp, c_vp,
                                     c_i32, c_i32, c_i64, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    ("dspark_test_set_first_wait_polls", None, [ctypes.c_uint32]),
    ("dspark_lattice_row_sample", c_i32, [c_vp, c_i32, c_i64, c_i32, c_i64, c_i64, c_vp, c_vp, c_vp, c_vp, c_i32,
                                          c_vp, c_i64, c_f32, c_f32, c_f32, c_f32, c_f32, c_vp, c_vp, c_vp, c_vp,
                                          c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    ("dspark_grouped_conv", c_i32, [c_vp, c_i32, c_i64, c_i64, c_i64, c_i32, c_i32, c_vp, c_vp, c_vp, c_i64, c_vp]),
    ("dspark_chain_select", c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_f32, c_f32, c_f32, c_vp, c_vp,
                                    c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    ("dspark_sample", c_i32, [c_vp, c_i32, c_i64, c_i32, c_i64, c_i64, c_vp, c_vp, c_i64, c_f32, c_f32, c_f32, c_f32,
                              c_f32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    ("dspark_dense_walk", c_i32, [c_vp, c_i32, c_i64, c_i32, c_i64, c_i64, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i64,
                                  c_vp, c_vp, c_vp, c_i32, c_i32, c_i64, c_f32, c_f32, c_f32, c_f32, c_vp, c_vp, c_vp,
                                  c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    ("dspark_verify", c_i32, [c_vp, c_i32, c_i64, c_i32, c_i64, c_i64, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_f32,
                              c_f32, c_f32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
]


class QRecord(ctypes.Structure):
    """dspark_qrecord: the proposal record (sparse or dense form)."""
    _fields_ = [("ids", c_vp), ("p", c_vp), ("n", c_vp), ("cap", c_i32), ("z", c_vp), ("ldz", c_i64),
                ("zmax", c_vp), ("wsum", c_vp), ("wcut", c_vp), ("icut", c_vp)]


class Penalties(ctypes.Structure):
    """dspark_penalties: the history and the repetition / presence penalties of a walk."""
    _fields_ = [("ids", c_vp), ("n", c_vp), ("cap", c_i32), ("repetition", c_f32), ("presence", c_f32)]


class DsparkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, self.code)}")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libdspark.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"libdspark.so is not built ({LIB}); run __graft_entry__.build()")
        handle = ctypes.CDLL(LIB)
        for name, res, args in SIGNATURES:
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(code: int, where: str) -> None:
    if code != 0:
        raise DsparkError(code, where)


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libdspark takes device tensors")
    return t.data_ptr()


def _dt(t) -> int:
    if t.dtype == torch.bfloat16:
        return DSPARK_BF16
    if t.dtype == torch.float32:
        return DSPARK_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _rows(t):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a row-major [rows, ld] tensor with unit column stride")
    return t.shape[0], t.stride(0)


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def read_status(status: torch.Tensor) -> int:
    return int(status.item())


def workspace(op: int, R: int, B: int, V: int, K: int = 0, device="cuda") -> torch.Tensor | None:
    n = int(lib().dspark_workspace_size(op, R, B, V, K))
    return torch.empty(n + 256, dtype=torch.uint8, device=device) if n else None


def _ws(t):
    """256-byte aligned (pointer, bytes) inside a uint8 workspace tensor."""
    if t is None:
        return None, 0
    p = t.data_ptr()
    off = (-p) % 256
    return p + off, max(0, t.numel() - off)


def dspark_status_string(code: int) -> str:
    return lib().dspark_status_string(code).decode()


def dspark_workspace_size(op: int, R: int, B: int, V: int, K: int = 0) -> int:
    return int(lib().dspark_workspace_size(op, R, B, V, K))


def dspark_d2t_check(d2t, V_t, require_injective=True, status=None, ws=None, stream=None):
    status = new_status(d2t.device) if status is None else status
    ws = workspace(OP_D2T_CHECK, 1, 1, V_t, 0, d2t.device) if ws is None else ws
    wp, wn = _ws(ws)
    _check(lib().dspark_d2t_check(_p(d2t), d2t.numel(), V_t, int(require_injective), wp, wn, _p(status),
                                  _stream(stream)), "dspark_d2t_check")
    return status


def dspark_d2t_check_noalloc(d2t, V_t, require_injective=True, status=None, stream=None):
    """dspark_d2t_check without a workspace (the library's static bitmap; V_t <= 2**20)."""
    status = new_status(d2t.device) if status is None else status
    _check(lib().dspark_d2t_check_noalloc(_p(d2t), d2t.numel(), V_t, int(require_injective), _p(status),
                                          _stream(stream)), "dspark_d2t_check_noalloc")
    return status


def dspark_topk(logits, B, K, *, R=None, V_d=None, row_start=None, mult=1.0, softcap=0.0, d2t=None, V_t=None,
                out=None, status=None, stream=None):
    rows, ld = _rows(logits)
    V_d = logits.shape[1] if V_d is None else V_d
    R = rows // B if R is None else R
    Kp = min(K, V_d)
    dev = logits.device
    if out is None:
        out = (torch.empty((R, B, Kp), dtype=torch.int32, device=dev),
               torch.empty((R, B, Kp), dtype=torch.int32, device=dev),
               torch.empty((R, B, Kp), dtype=torch.float32, device=dev))
    status = new_status(dev) if status is None else status
    V_t = (V_d if d2t is None else V_t) if V_t is None else V_t
    _check(lib().dspark_topk(_p(logits), _dt(logits), R, B, V_d, ld, _p(row_start), K, mult, softcap, _p(d2t), V_t,
                             _p(out[0]), _p(out[1]), _p(out[2]), _p(status), _stream(stream)), "dspark_topk")
    return out + (status,)


def dspark_lattice_score(cand_tgt, prev, E, W, *, hidden=None, g=None, row_start=None, out=None, status=None,
                         stream=None):
    R, B, K = cand_tgt.shape
    V_t, rank = E.shape
    dev = cand_tgt.device
    if out is None:
        out = (torch.empty((R, B, K, K), dtype=torch.float32, device=dev),
               torch.empty((R, B), dtype=torch.float32, device=dev))
    status = new_status(dev) if status is None else status
    if hidden is not None:
        _, ldh = _rows(hidden)
        H, hdt = hidden.shape[1], _dt(hidden)
    else:
        ldh, H, hdt = 0, 0, DSPARK_BF16
    _check(lib().dspark_lattice_score(_p(cand_tgt), _p(prev), R, B, K, _p(E), _p(W), _dt(E), V_t, rank, _p(hidden),
                                      _p(g), hdt, H, ldh, _p(row_start), _p(out[0]), _p(out[1]), _p(status),
                                      _stream(stream)), "dspark_lattice_score")
    return out + (status,)


def _qrec_sparse(ids, p, n):
    return QRecord(ids=_p(ids), p=_p(p), n=_p(n), cap=ids.shape[-1])


def dspark_chain_select(cand_val, trans, cand_tgt, mode="maxsum", *, temperature=0.0, top_p=1.0, seed=None,
                        step=None, record=True, q=None, out=None, status=None, stream=None, temperature_r=None,
                        top_p_r=None, min_p=0.0, min_p_r=None, history=None, repetition=1.0, presence=0.0):
    """temperature_r / top_p_r: optional [R] float32 per-request values (a mixed greedy/sampled
    batch; temperature <= 0 walks greedily) that replace the scalars in the sampled mode."""
    R, B, K = cand_val.shape
    dev = cand_val.device
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    if out is None:
        out = (torch.empty((R, B), dtype=torch.int32, device=dev), torch.empty((R, B), dtype=torch.int32, device=dev),
               torch.empty((R,), dtype=torch.float32, device=dev))
    status = new_status(dev) if status is None else status
    qt = ()
    if m != DSPARK_SAMPLE:
        q = None
    elif q is not None:                                     # caller's sparse record (ids, p, n)
        qt = tuple(q)
        q = _qrec_sparse(*qt)
    elif record:
        qt = (torch.full((R, B, K), -1, dtype=torch.int32, device=dev), torch.zeros((R, B, K), dtype=torch.float32,
                                                                                   device=dev),
              torch.zeros((R, B), dtype=torch.int32, device=dev))
        q = _qrec_sparse(*qt)
    pen = None
    if history is not None:                                 # (ids [R, cap] int32, n [R] int32)
        ids, nh = history
        pen = Penalties(_p(ids), _p(nh), ids.shape[1], repetition, presence)
    _check(lib().dspark_chain_select(_p(cand_val), _p(trans), _p(cand_tgt), R, B, K, m, temperature, top_p, min_p,
                                     _p(temperature_r), _p(top_p_r), _p(min_p_r),
                                     ctypes.byref(pen) if pen is not None else None, _p(seed),
                                     _p(step), _p(out[0]), _p(out[1]), _p(out[2]),
                                     ctypes.byref(q) if q is not None else None, _p(status), _stream(stream)),
           "dspark_chain_select")
    return out + qt + (status,)


def dspark_lattice_chain(cand_val, cand_tgt, prev, E, W, mode="maxsum", *, hidden=None, g=None, row_start=None,
                         trans=None, gate=None, out=None, status=None, stream=None):
    """Lattice + greedy chain (max-sum or walk) in one call; trans/gate are written only if given."""
    R, B, K = cand_tgt.shape
    V_t, rank = E.shape
    dev = cand_tgt.device
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    if out is None:
        out = (torch.empty((R, B), dtype=torch.int32, device=dev), torch.empty((R, B), dtype=torch.int32, device=dev),
               torch.empty((R,), dtype=torch.float32, device=dev))
    status = new_status(dev) if status is None else status
    if hidden is not None:
        _, ldh = _rows(hidden)
        H, hdt = hidden.shape[1], _dt(hidden)
    else:
        ldh, H, hdt = 0, 0, DSPARK_BF16
    _check(lib().dspark_lattice_chain(_p(cand_val), _p(cand_tgt), _p(prev), R, B, K, _p(E), _p(W), _dt(E), V_t, rank,
                                      _p(hidden), _p(g), hdt, H, ldh, _p(row_start), m, _p(trans), _p(gate),
                                      _p(out[0]), _p(out[1]), _p(out[2]), _p(status), _stream(stream)),
           "dspark_lattice_chain")
    return out + (status,)


def dspark_lattice_row_sample(logits, B, cand_draft, cand_val, trans, *, R=None, V_d=None, row_start=None, d2t=None,
                              V_t=None, mult=1.0, softcap=0.0, temperature=1.0, top_p=1.0, min_p=0.0, seed=None,
                              step=None, q=None, out=None, ws=None, status=None, stream=None):
    """The lattice-row branch: returns (out_tgt [R, B], out_idx [R, B], n_drafted [R], status)."""
    rows, ld = _rows(logits)
    V_d = logits.shape[1] if V_d is None else V_d
    R = cand_draft.shape[0] if R is None else R
    K = cand_draft.shape[2]
    dev = logits.device
    V_t = (V_d if d2t is None else V_t) if V_t is None else V_t
    if out is None:
        out = (torch.empty((R, B), dtype=torch.int32, device=dev), torch.empty((R, B), dtype=torch.int32, device=dev),
               torch.empty((R,), dtype=torch.int32, device=dev))
    status = new_status(dev) if status is None else status
    ws = workspace(OP_LATTICE_ROW, R, B, V_d, K, dev) if ws is None else ws
    wp, wn = _ws(ws)
    qr = _qrec_any(q)
    _check(lib().dspark_lattice_row_sample(_p(logits), _dt(logits), R, B, V_d, ld, _p(row_start), _p(cand_draft),
                                           _p(cand_val), _p(trans), K, _p(d2t), V_t, mult, softcap, temperature, top_p,
                                           min_p, _p(seed), _p(step), _p(out[0]), _p(out[1]), _p(out[2]),
                                           ctypes.byref(qr) if qr is not None else None, wp, wn, _p(status),
                                           _stream(stream)), "dspark_lattice_row_sample")
    return out + (status,)


def dspark_grouped_conv(x, k, block, *, out=None, stream=None):
    """DFlash-2 grouped dynamic convolution over packed block rows: x [N, C] (bf16/f32),
    k [N, G, L] float32 taps, block [N] int32 -> y [N, C] float32."""
    N, ldx = _rows(x)
    C = x.shape[1]
    G, L = k.shape[1], k.shape[2]
    y = out if out is not None else torch.empty((N, C), dtype=torch.float32, device=x.device)
    _, ldy = _rows(y)
    _check(lib().dspark_grouped_conv(_p(x), _dt(x), N, C, ldx, G, L, _p(k), _p(block), _p(y), ldy, _stream(stream)),
           "dspark_grouped_conv")
    return y


def dspark_test_set_first_wait_polls(polls: int) -> None:
    """Test hook: poll limit of the first tensor-core completion wait (0xFFFFFFFF: default)."""
    lib().dspark_test_set_first_wait_polls(polls)


def dense_record(rows: int, V: int, device="cuda"):
    """Allocates a dense proposal record: (z [rows, V] f32, zmax, wsum (f64), wcut, icut)."""
    return (torch.empty((rows, V), dtype=torch.float32, device=device),
            torch.empty((rows,), dtype=torch.float32, device=device),
            torch.empty((rows,), dtype=torch.float64, device=device),
            torch.empty((rows,), dtype=torch.float32, device=device),
            torch.empty((rows,), dtype=torch.int32, device=device))


def _qrec_dense(z, zmax, wsum, wcut, icut):
    return QRecord(z=_p(z), ldz=z.stride(0), zmax=_p(zmax), wsum=_p(wsum), wcut=_p(wcut), icut=_p(icut))


def _qrec_any(q):
    if q is None:
        return None
    if len(q) == 3:
        return _qrec_sparse(*q)
    return _qrec_dense(*q)


def dspark_sample(logits, B, *, R=None, V_d=None, row_start=None, d2t=None, V_t=None, mult=1.0, softcap=0.0,
                  temperature=1.0, top_p=1.0, seed=None, step=None, q=None, out=None, ws=None, status=None,
                  stream=None, temperature_r=None, top_p_r=None, min_p=0.0, min_p_r=None):
    """temperature_r / top_p_r / min_p_r: optional [R] float32 per-request values (a mixed batch)."""
    rows, ld = _rows(logits)
    V_d = logits.shape[1] if V_d is None else V_d
    R = rows // B if R is None else R
    dev = logits.device
    V_t = (V_d if d2t is None else V_t) if V_t is None else V_t
    if out is None:
        out = (torch.empty((R, B), dtype=torch.int32, device=dev), torch.empty((R, B), dtype=torch.int32, device=dev))
    status = new_status(dev) if status is None else status
    ws = workspace(OP_SAMPLE, R, B, V_d, 0, dev) if ws is None else ws
    wp, wn = _ws(ws)
    qr = _qrec_any(q)
    _check(lib().dspark_sample(_p(logits), _dt(logits), R, B, V_d, ld, _p(row_start), _p(d2t), V_t, mult, softcap,
                               temperature, top_p, min_p, _p(temperature_r), _p(top_p_r), _p(min_p_r), _p(seed),
                               _p(step), _p(out[0]), _p(out[1]),
                               ctypes.byref(qr) if qr is not None else None, wp, wn, _p(status), _stream(stream)),
           "dspark_sample")
    return out + (status,)


def dspark_dense_walk(logits, B, prev, E, W, *, R=None, V_d=None, row_start=None, d2t=None, hidden=None, g=None,
                      mult=1.0, softcap=0.0, temperature=0.0, top_p=1.0, seed=None, step=None, q=None, out=None,
                      ws=None, status=None, stream=None):
    rows, ld = _rows(logits)
    V_d = logits.shape[1] if V_d is None else V_d
    R = rows // B if R is None else R
    V_t, rank = E.shape
    dev = logits.device
    if out is None:
        out = (torch.empty((R, B), dtype=torch.int32, device=dev), torch.empty((R, B), dtype=torch.int32, device=dev))
    status = new_status(dev) if status is None else status
    ws = workspace(OP_DENSE_WALK, R, B, V_d, 0, dev) if ws is None else ws
    wp, wn = _ws(ws)
    if hidden is not None:
        _, ldh = _rows(hidden)
        H, hdt = hidden.shape[1], _dt(hidden)
    else:
        ldh, H, hdt = 0, 0, DSPARK_BF16
    qr = _qrec_any(q)
    _check(lib().dspark_dense_walk(_p(logits), _dt(logits), R, B, V_d, ld, _p(row_start), _p(prev), _p(E), _p(W),
                                   _dt(E), rank, V_t, _p(d2t), _p(hidden), _p(g), hdt, H, ldh, mult, softcap,
                                   temperature, top_p, _p(seed), _p(step), _p(out[0]), _p(out[1]),
                                   ctypes.byref(qr) if qr is not None else None, wp, wn, _p(status),
                                   _stream(stream)), "dspark_dense_walk")
    return out + (status,)


def dspark_verify(tgt_logits, B, draft_tgt, n_draft, q, *, V_q=None, q_d2t=None, R=None, row_start=None,
                  temperature=1.0, top_p=1.0, vseed=None, step=None, out=None, ws=None, status=None, stream=None,
                  temperature_r=None, top_p_r=None, min_p=0.0, min_p_r=None):
    """temperature_r / top_p_r / min_p_r: optional [R] float32 per-request values (a mixed batch)."""
    rows, ld = _rows(tgt_logits)
    V_t = tgt_logits.shape[1]
    R = draft_tgt.shape[0] if R is None else R
    dev = tgt_logits.device
    if out is None:
        out = (torch.empty((R, B + 1), dtype=torch.int32, device=dev), torch.empty((R,), dtype=torch.int32, device=dev),
               torch.empty((R, B + 1), dtype=torch.float32, device=dev))
    status = new_status(dev) if status is None else status
    ws = workspace(OP_VERIFY, R, B, V_t, 0, dev) if ws is None else ws
    wp, wn = _ws(ws)
    qr = _qrec_any(q)
    if V_q is None:
        V_q = q[0].shape[1] if (q is not None and len(q) == 5) else V_t
    _check(lib().dspark_verify(_p(tgt_logits), _dt(tgt_logits), R, B, V_t, ld, _p(row_start), _p(draft_tgt),
                               _p(n_draft), ctypes.byref(qr) if qr is not None else None, V_q, _p(q_d2t),
                               temperature, top_p, min_p, _p(temperature_r), _p(top_p_r), _p(min_p_r),
                               _p(vseed), _p(step), _p(out[0]), _p(out[1]), _p(out[2]), wp, wn, _p(status),
                               _stream(stream)), "dspark_verify")
    return out + (status,)
