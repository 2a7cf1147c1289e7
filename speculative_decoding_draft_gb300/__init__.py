"""DSpark per-step speculative-decoding hot path on one GB300 (sm_103a).

Python binding of ``libdspark.so`` (see ``include/dspark.h``).  The functions
here only marshal arguments: they check tensor placement, dtypes and shapes,
allocate outputs and workspaces with torch on the tensors' device, and call the
C ABI on the current CUDA stream.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback.  If the library has
not been built, every call raises ``DsparkUnavailable``.

Method: "DSpark: Confidence-Scheduled Speculative Decoding with
Semi-Autoregressive Generation" (S2.1 acceptance rule, S3.1 Markov head,
S3.2.2 Algorithm 1).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "DsparkError", "DsparkUnavailable", "lib", "library_path", "draft_markov_sample", "schedule_survival",
    "verify_ragged", "check", "status_string", "draft_workspace_bytes", "schedule_workspace_bytes",
    "verify_workspace_bytes", "F32", "BF16", "FLAG_FORCE_SIMT", "FLAG_W_PACKED", "FLAG_SPARE_SM", "STATUS_NAMES", "Dims",
    "PackedProjection", "pack_projection", "packed_projection_bytes", "verify_markov",
    "verify_markov_workspace_bytes",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
# DSPARK_LIBRARY selects another build of the same library (the bounds-checked one in tests)
_LIB_PATH = os.environ.get("DSPARK_LIBRARY") or os.path.join(_HERE, "libdspark.so")

F32, BF16 = 0, 1
FLAG_FORCE_SIMT = 1
FLAG_W_PACKED = 2
FLAG_SPARE_SM = 4
FLAG_TEST_BARRIER_TIMEOUT = 8   # failure-path test hook of the tensor-core draft (see include/dspark.h)

STATUS_NAMES = {
    0: "DSPARK_OK", 1: "DSPARK_ERR_NULL", 2: "DSPARK_ERR_DIMS", 3: "DSPARK_ERR_DTYPE",
    4: "DSPARK_ERR_TEMPERATURE", 5: "DSPARK_ERR_SPS_TOO_SHORT", 6: "DSPARK_ERR_OFFSETS",
    7: "DSPARK_ERR_TOKEN_RANGE", 8: "DSPARK_ERR_LENGTHS", 9: "DSPARK_ERR_CONFIDENCE",
    10: "DSPARK_ERR_WORKSPACE", 11: "DSPARK_ERR_DEVICE_TIMEOUT", 12: "DSPARK_ERR_CUDA",
    13: "DSPARK_ERR_UNSUPPORTED", 14: "DSPARK_ERR_BOUNDS",
}

EXPORTED_SYMBOLS = [
    "dspark_draft_workspace_bytes", "dspark_draft_markov_sample", "dspark_draft_markov_sample_confidence",
    "dspark_draft_rnn_workspace_bytes", "dspark_draft_rnn_sample", "dspark_draft_packed_projection_bytes",
    "dspark_draft_pack_projection", "dspark_schedule_workspace_bytes",
    "dspark_schedule_survival", "dspark_schedule_survival_noalloc", "dspark_schedule_capacity",
    "dspark_schedule_topk", "dspark_schedule_threshold", "dspark_verify_workspace_bytes",
    "dspark_verify_ragged", "dspark_verify_markov_workspace_bytes", "dspark_verify_markov",
    "dspark_status_string", "dspark_check", "dspark_version",
]


class DsparkUnavailable(RuntimeError):
    pass


class DsparkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS_NAMES.get(code, f"DSPARK_ERR_{code}")
        super().__init__(f"{where}: {self.name}")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("K_max", ctypes.c_int64), ("V", ctypes.c_int64),
                ("rank", ctypes.c_int64), ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32)]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libdspark.so (raises DsparkUnavailable when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise DsparkUnavailable(f"{_LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(_LIB_PATH)
    P, i64, u64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    st = ctypes.c_int
    L.dspark_draft_workspace_bytes.argtypes = [Dims]
    L.dspark_draft_workspace_bytes.restype = sz
    L.dspark_draft_packed_projection_bytes.argtypes = [i64, i64]
    L.dspark_draft_packed_projection_bytes.restype = sz
    L.dspark_draft_pack_projection.argtypes = [P, Dims, P, sz, P]
    L.dspark_draft_pack_projection.restype = st
    L.dspark_draft_markov_sample.argtypes = [P, P, P, P, P, P, u64, Dims, P, P, P, P, P, sz, P, P]
    L.dspark_draft_markov_sample.restype = st
    L.dspark_draft_markov_sample_confidence.argtypes = [P, P, P, P, P, P, u64, Dims, P, P, P, P, P, P, P, P, sz, P,
                                                         P]
    L.dspark_draft_markov_sample_confidence.restype = st
    L.dspark_draft_rnn_workspace_bytes.argtypes = [Dims]
    L.dspark_draft_rnn_workspace_bytes.restype = sz
    L.dspark_draft_rnn_sample.argtypes = [P, P, P, P, P, P, P, P, u64, Dims, P, P, P, P, P, sz, P, P]
    L.dspark_draft_rnn_sample.restype = st
    L.dspark_schedule_workspace_bytes.argtypes = [i64, i64]
    L.dspark_schedule_workspace_bytes.restype = sz
    L.dspark_schedule_survival.argtypes = [P, P, P, i64, i64, i64, P, P, P, P, P, P, sz, P, P]
    L.dspark_schedule_survival.restype = st
    L.dspark_schedule_survival_noalloc.argtypes = [P, P, P, i64, i64, i64, P, P, P, P, P, P, P]
    L.dspark_schedule_survival_noalloc.restype = st
    L.dspark_schedule_capacity.argtypes = [P, P, P, i64, i64, i64, P, P, P, P, P, sz, P, P]
    L.dspark_schedule_capacity.restype = st
    L.dspark_schedule_topk.argtypes = [P, P, P, i64, i64, P, P, P, P, P, sz, P, P]
    L.dspark_schedule_topk.restype = st
    L.dspark_schedule_threshold.argtypes = [P, P, ctypes.c_float, ctypes.c_int32, i64, i64, P, P, P, P, P, P]
    L.dspark_schedule_threshold.restype = st
    L.dspark_verify_workspace_bytes.argtypes = [i64, i64]
    L.dspark_verify_workspace_bytes.restype = sz
    L.dspark_verify_ragged.argtypes = [P, P, P, P, P, P, P, u64, Dims, P, P, P, sz, P, P]
    L.dspark_verify_ragged.restype = st
    L.dspark_verify_markov_workspace_bytes.argtypes = [Dims]
    L.dspark_verify_markov_workspace_bytes.restype = sz
    L.dspark_verify_markov.argtypes = [P, P, P, P, P, P, P, P, P, P, P, u64, Dims, P, P, P, sz, P, P]
    L.dspark_verify_markov.restype = st
    L.dspark_status_string.argtypes = [st]
    L.dspark_status_string.restype = ctypes.c_char_p
    L.dspark_check.argtypes = [P, P]
    L.dspark_check.restype = st
    L.dspark_version.argtypes = []
    L.dspark_version.restype = ctypes.c_int
    _lib = L
    return L


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]) -> torch.Tensor:
    if ws is not None and ws.numel() >= nbytes and ws.data_ptr() % 256 == 0:
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _raise(code: int, where: str):
    if code != 0:
        raise DsparkError(code, where)


def status_string(code: int) -> str:
    return lib().dspark_status_string(int(code)).decode()


def check(dev_status: torch.Tensor, stream=None) -> str:
    """Synchronise, read and reset the device status word; returns its name."""
    code = lib().dspark_check(_ptr(dev_status), _stream(stream))
    return STATUS_NAMES.get(code, f"DSPARK_ERR_{code}")


def draft_workspace_bytes(B: int, K_max: int, V: int, rank: int, dtype: int = BF16, flags: int = 0) -> int:
    return int(lib().dspark_draft_workspace_bytes(Dims(B, K_max, V, rank, dtype, flags)))


def packed_projection_bytes(rank: int, V: int) -> int:
    return int(lib().dspark_draft_packed_projection_bytes(rank, V))


class PackedProjection:
    """W2 in the packed tensor-core layout (dspark_draft_pack_projection): a uint8 device
    tensor plus the shape it was packed from."""

    def __init__(self, data: torch.Tensor, rank: int, V: int):
        self.data, self.rank, self.V = data, rank, V
        self.dtype = torch.bfloat16
        self.device = data.device


def pack_projection(W, *, stream=None) -> PackedProjection:
    """Pack W2 [rank, V] bfloat16 once for the tensor-core draft path."""
    _dev(W, "W", torch.bfloat16)
    rank, V = W.shape
    nbytes = packed_projection_bytes(rank, V)
    if nbytes == 0:
        raise DsparkError(13, "dspark_draft_pack_projection")
    data = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    code = lib().dspark_draft_pack_projection(_ptr(W), Dims(1, 1, V, rank, BF16, 0), _ptr(data),
                                             ctypes.c_size_t(nbytes), _stream(stream))
    _raise(code, "dspark_draft_pack_projection")
    return PackedProjection(data, rank, V)


def schedule_workspace_bytes(B: int, K_max: int) -> int:
    return int(lib().dspark_schedule_workspace_bytes(B, K_max))


def verify_workspace_bytes(B: int, V: int) -> int:
    return int(lib().dspark_verify_workspace_bytes(B, V))


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def draft_markov_sample(U, E, W, anchor, K_r, temperature, seed: int, *, want_logits: bool = True,
                        want_lse: bool = True, want_tok_logit: bool = True, force_simt: bool = False,
                        spare_sm: bool = False,
                        conf_h=None, conf_w=None, out: Optional[dict] = None,
                        workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                        stream=None) -> dict:
    """Markov-head draft sampling (C ABI dspark_draft_markov_sample).

    U [B,K_max,V], E [V,rank], W [rank,V] (float32 or bfloat16, one dtype) or a
    PackedProjection of W (bfloat16, tensor-core path);
    anchor, K_r [B] int32; temperature [B] float32.  Returns a dict with
    draft_tok [B,K_max] int32, draft_logits (U's dtype) or None, draft_lse
    [B,K_max] float32 or None, draft_tok_logit [B,K_max] float32 (the drawn tokens'
    logits) or None, and the status / workspace tensors used.
    spare_sm leaves one SM free of the tensor-core path's persistent kernel, for a
    kernel on another stream (the scheduler) to run beside it.
    With conf_h [B,K_max] float32 (the backbone term of the confidence head) and
    conf_w [rank] float32 (its weights on the Markov embedding), the call is
    dspark_draft_markov_sample_confidence and also returns conf [B,K_max] float32.
    """
    dt = _dtype_code(_dev(U, "U"))
    B, K_max, V = U.shape
    rank = E.shape[1]
    _dev(E, "E", U.dtype, (V, rank))
    flags = (FLAG_FORCE_SIMT if force_simt else 0) | (FLAG_SPARE_SM if spare_sm else 0)
    if isinstance(W, PackedProjection):
        if (W.rank, W.V) != (rank, V) or W.device != U.device or U.dtype != W.dtype:
            raise ValueError(f"packed projection of shape ({W.rank}, {W.V}) does not fit U/E")
        flags |= FLAG_W_PACKED
        W = W.data
    else:
        _dev(W, "W", U.dtype, (rank, V))
    _dev(anchor, "anchor", torch.int32, (B,))
    _dev(K_r, "K_r", torch.int32, (B,))
    _dev(temperature, "temperature", torch.float32, (B,))
    dev = U.device
    out = {} if out is None else out
    tok = out.get("draft_tok")
    if tok is None:
        tok = torch.empty(B, K_max, dtype=torch.int32, device=dev)
    logits = out.get("draft_logits") if want_logits else None
    if want_logits and logits is None:
        logits = torch.empty_like(U)
    lse = out.get("draft_lse") if want_lse else None
    if want_lse and lse is None:
        lse = torch.empty(B, K_max, dtype=torch.float32, device=dev)
    zx = out.get("draft_tok_logit") if want_tok_logit else None
    if want_tok_logit and zx is None:
        zx = torch.empty(B, K_max, dtype=torch.float32, device=dev)
    status = new_status(dev) if status is None else status
    nbytes = draft_workspace_bytes(B, K_max, V, rank, dt, flags)
    ws = _workspace(nbytes, dev, workspace)
    dims = Dims(B, K_max, V, rank, dt, flags)
    if (conf_h is None) != (conf_w is None):
        raise ValueError("conf_h and conf_w go together")
    conf = None
    if conf_h is None:
        code = lib().dspark_draft_markov_sample(_ptr(U), _ptr(E), _ptr(W), _ptr(anchor), _ptr(K_r),
                                                _ptr(temperature), ctypes.c_uint64(seed), dims, _ptr(tok),
                                                _ptr(logits), _ptr(lse), _ptr(zx), _ptr(ws),
                                                ctypes.c_size_t(ws.numel()), _ptr(status), _stream(stream))
        _raise(code, "dspark_draft_markov_sample")
    else:
        _dev(conf_h, "conf_h", torch.float32, (B, K_max))
        _dev(conf_w, "conf_w", torch.float32, (rank,))
        conf = out.get("conf")
        if conf is None:
            conf = torch.empty(B, K_max, dtype=torch.float32, device=dev)
        code = lib().dspark_draft_markov_sample_confidence(
            _ptr(U), _ptr(E), _ptr(W), _ptr(anchor), _ptr(K_r), _ptr(temperature), ctypes.c_uint64(seed), dims,
            _ptr(conf_h), _ptr(conf_w), _ptr(tok), _ptr(logits), _ptr(lse), _ptr(zx), _ptr(conf), _ptr(ws),
            ctypes.c_size_t(ws.numel()), _ptr(status), _stream(stream))
        _raise(code, "dspark_draft_markov_sample_confidence")
    return dict(draft_tok=tok, draft_logits=logits, draft_lse=lse, draft_tok_logit=zx, conf=conf, status=status,
                workspace=ws)


def draft_rnn_sample(U, E, W, rnn_W, rnn_x, anchor, K_r, temperature, seed: int, *, want_logits: bool = True,
                     want_lse: bool = True, want_tok_logit: bool = True, out: Optional[dict] = None,
                     workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                     stream=None) -> dict:
    """RNN-head draft sampling (C ABI dspark_draft_rnn_sample).

    U [B,K_max,V], E [V,rank], W [rank,V], rnn_W [3 rank, 2 rank] (one dtype); rnn_x
    [B,K_max,3 rank] float32; anchor, K_r [B] int32; temperature [B] float32.  Returns
    draft_tok, draft_logits, draft_lse, draft_tok_logit as draft_markov_sample does.
    """
    dt = _dtype_code(_dev(U, "U"))
    B, K_max, V = U.shape
    rank = E.shape[1]
    _dev(E, "E", U.dtype, (V, rank))
    _dev(W, "W", U.dtype, (rank, V))
    _dev(rnn_W, "rnn_W", U.dtype, (3 * rank, 2 * rank))
    _dev(rnn_x, "rnn_x", torch.float32, (B, K_max, 3 * rank))
    _dev(anchor, "anchor", torch.int32, (B,))
    _dev(K_r, "K_r", torch.int32, (B,))
    _dev(temperature, "temperature", torch.float32, (B,))
    dev = U.device
    out = {} if out is None else out
    tok = _out(out, "draft_tok", (B, K_max), torch.int32, dev)
    logits = (out.get("draft_logits") if out.get("draft_logits") is not None else torch.empty_like(U)) \
        if want_logits else None
    lse = _out(out, "draft_lse", (B, K_max), torch.float32, dev) if want_lse else None
    zx = _out(out, "draft_tok_logit", (B, K_max), torch.float32, dev) if want_tok_logit else None
    status = new_status(dev) if status is None else status
    dims = Dims(B, K_max, V, rank, dt, 0)
    ws = _workspace(lib().dspark_draft_rnn_workspace_bytes(dims), dev, workspace)
    code = lib().dspark_draft_rnn_sample(_ptr(U), _ptr(E), _ptr(W), _ptr(rnn_W), _ptr(rnn_x), _ptr(anchor),
                                         _ptr(K_r), _ptr(temperature), ctypes.c_uint64(seed), dims, _ptr(tok),
                                         _ptr(logits), _ptr(lse), _ptr(zx), _ptr(ws), ctypes.c_size_t(ws.numel()),
                                         _ptr(status), _stream(stream))
    _raise(code, "dspark_draft_rnn_sample")
    return dict(draft_tok=tok, draft_logits=logits, draft_lse=lse, draft_tok_logit=zx, status=status, workspace=ws)


def schedule_survival(conf, K_r, sps, *, out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                      status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Hardware-aware prefix scheduler (C ABI dspark_schedule_survival).

    conf [B,K_max] float32, K_r [B] int32, sps float64 (CUDA).  Returns ell [B],
    tgt_off [B+1] (int32), theta_best [1] float64, b_star [1] int64 and survival
    [B,K_max] float32.
    """
    _dev(conf, "conf", torch.float32)
    B, K_max = conf.shape
    _dev(K_r, "K_r", torch.int32, (B,))
    _dev(sps, "sps", torch.float64)
    dev = conf.device
    out = {} if out is None else out
    ell = out.get("ell") if out.get("ell") is not None else torch.empty(B, dtype=torch.int32, device=dev)
    off = out.get("tgt_off") if out.get("tgt_off") is not None else torch.empty(B + 1, dtype=torch.int32, device=dev)
    th = out.get("theta_best") if out.get("theta_best") is not None else torch.empty(1, dtype=torch.float64, device=dev)
    bs = out.get("b_star") if out.get("b_star") is not None else torch.empty(1, dtype=torch.int64, device=dev)
    surv = out.get("survival") if out.get("survival") is not None else torch.empty(B, K_max, dtype=torch.float32,
                                                                                   device=dev)
    status = new_status(dev) if status is None else status
    ws = _workspace(schedule_workspace_bytes(B, K_max), dev, workspace)
    code = lib().dspark_schedule_survival(_ptr(conf), _ptr(K_r), _ptr(sps), sps.numel(), B, K_max, _ptr(ell),
                                          _ptr(off), _ptr(th), _ptr(bs), _ptr(surv), _ptr(ws),
                                          ctypes.c_size_t(ws.numel()), _ptr(status), _stream(stream))
    _raise(code, "dspark_schedule_survival")
    return dict(ell=ell, tgt_off=off, theta_best=th, b_star=bs, survival=surv, status=status, workspace=ws)


def _out(out, key, shape, dtype, dev):
    t = out.get(key)
    return t if t is not None else torch.empty(shape, dtype=dtype, device=dev)


def schedule_capacity(conf, K_r, sps, *, out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                      status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Capacity of the asynchronous scheduler (C ABI dspark_schedule_capacity).

    conf [B,K_max] float32, K_r [B] int32, sps float64 (CUDA).  Returns capacity [1]
    int32 (admitted draft tokens at the global maximum of Theta), theta_best [1] float64
    and the retrospective lengths ell [B] / tgt_off [B+1] of that admission.
    """
    _dev(conf, "conf", torch.float32)
    B, K_max = conf.shape
    _dev(K_r, "K_r", torch.int32, (B,))
    _dev(sps, "sps", torch.float64)
    dev = conf.device
    out = {} if out is None else out
    cap = _out(out, "capacity", (1,), torch.int32, dev)
    th = _out(out, "theta_best", (1,), torch.float64, dev)
    ell = _out(out, "ell", (B,), torch.int32, dev)
    off = _out(out, "tgt_off", (B + 1,), torch.int32, dev)
    status = new_status(dev) if status is None else status
    ws = _workspace(schedule_workspace_bytes(B, K_max), dev, workspace)
    code = lib().dspark_schedule_capacity(_ptr(conf), _ptr(K_r), _ptr(sps), sps.numel(), B, K_max, _ptr(cap),
                                          _ptr(th), _ptr(ell), _ptr(off), _ptr(ws), ctypes.c_size_t(ws.numel()),
                                          _ptr(status), _stream(stream))
    _raise(code, "dspark_schedule_capacity")
    return dict(capacity=cap, theta_best=th, ell=ell, tgt_off=off, status=status, workspace=ws)


def schedule_topk(conf, K_r, capacity, *, out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                  status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Dynamic top-K admission (C ABI dspark_schedule_topk); capacity is a CUDA int32 [1] tensor."""
    _dev(conf, "conf", torch.float32)
    B, K_max = conf.shape
    _dev(K_r, "K_r", torch.int32, (B,))
    _dev(capacity, "capacity", torch.int32, (1,))
    dev = conf.device
    out = {} if out is None else out
    ell = _out(out, "ell", (B,), torch.int32, dev)
    off = _out(out, "tgt_off", (B + 1,), torch.int32, dev)
    bs = _out(out, "b_star", (1,), torch.int64, dev)
    surv = _out(out, "survival", (B, K_max), torch.float32, dev)
    status = new_status(dev) if status is None else status
    ws = _workspace(schedule_workspace_bytes(B, K_max), dev, workspace)
    code = lib().dspark_schedule_topk(_ptr(conf), _ptr(K_r), _ptr(capacity), B, K_max, _ptr(ell), _ptr(off),
                                      _ptr(bs), _ptr(surv), _ptr(ws), ctypes.c_size_t(ws.numel()), _ptr(status),
                                      _stream(stream))
    _raise(code, "dspark_schedule_topk")
    return dict(ell=ell, tgt_off=off, b_star=bs, survival=surv, status=status, workspace=ws)


THRESHOLD_CONFIDENCE, THRESHOLD_SURVIVAL = 0, 1


def schedule_threshold(conf, K_r, threshold: float, mode: int = THRESHOLD_CONFIDENCE, *,
                       out: Optional[dict] = None, status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Static-threshold lengths (C ABI dspark_schedule_threshold)."""
    _dev(conf, "conf", torch.float32)
    B, K_max = conf.shape
    _dev(K_r, "K_r", torch.int32, (B,))
    dev = conf.device
    out = {} if out is None else out
    ell = _out(out, "ell", (B,), torch.int32, dev)
    off = _out(out, "tgt_off", (B + 1,), torch.int32, dev)
    bs = _out(out, "b_star", (1,), torch.int64, dev)
    surv = _out(out, "survival", (B, K_max), torch.float32, dev)
    status = new_status(dev) if status is None else status
    code = lib().dspark_schedule_threshold(_ptr(conf), _ptr(K_r), float(threshold), int(mode), B, K_max,
                                           _ptr(ell), _ptr(off), _ptr(bs), _ptr(surv), _ptr(status),
                                           _stream(stream))
    _raise(code, "dspark_schedule_threshold")
    return dict(ell=ell, tgt_off=off, b_star=bs, survival=surv, status=status)


def verify_ragged(draft_logits, tgt_logits, tgt_off, ell, draft_tok, temperature, seed: int, *,
                  draft_lse=None, out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                  status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Ragged rejection-sampling verification (C ABI dspark_verify_ragged).

    draft_logits [B,K_max,V], tgt_logits [sum(ell+1),V] (one dtype), tgt_off
    [B+1], ell [B], draft_tok [B,K_max] int32, temperature [B] float32,
    draft_lse [B,K_max] float32 or None.  Returns n_acc [B] and out_tok
    [B,K_max+1] (int32).
    """
    dt = _dtype_code(_dev(draft_logits, "draft_logits"))
    B, K_max, V = draft_logits.shape
    _dev(tgt_logits, "tgt_logits", draft_logits.dtype)
    if tgt_logits.dim() != 2 or tgt_logits.shape[1] != V:
        raise ValueError("tgt_logits must be [rows, V]")
    _dev(tgt_off, "tgt_off", torch.int32, (B + 1,))
    _dev(ell, "ell", torch.int32, (B,))
    _dev(draft_tok, "draft_tok", torch.int32, (B, K_max))
    _dev(temperature, "temperature", torch.float32, (B,))
    if draft_lse is not None:
        _dev(draft_lse, "draft_lse", torch.float32, (B, K_max))
    dev = draft_logits.device
    out = {} if out is None else out
    n_acc = out.get("n_acc") if out.get("n_acc") is not None else torch.empty(B, dtype=torch.int32, device=dev)
    out_tok = out.get("out_tok") if out.get("out_tok") is not None else torch.empty(B, K_max + 1, dtype=torch.int32,
                                                                                    device=dev)
    status = new_status(dev) if status is None else status
    ws = _workspace(verify_workspace_bytes(B, V), dev, workspace)
    dims = Dims(B, K_max, V, 0, dt, 0)
    code = lib().dspark_verify_ragged(_ptr(draft_logits), _ptr(draft_lse), _ptr(tgt_logits), _ptr(tgt_off),
                                      _ptr(ell), _ptr(draft_tok), _ptr(temperature), ctypes.c_uint64(seed), dims,
                                      _ptr(n_acc), _ptr(out_tok), _ptr(ws), ctypes.c_size_t(ws.numel()),
                                      _ptr(status), _stream(stream))
    _raise(code, "dspark_verify_ragged")
    return dict(n_acc=n_acc, out_tok=out_tok, status=status, workspace=ws)


def verify_markov_workspace_bytes(B: int, K_max: int, V: int, rank: int, packed: bool = True) -> int:
    return int(lib().dspark_verify_markov_workspace_bytes(Dims(B, K_max, V, rank, BF16,
                                                                FLAG_W_PACKED if packed else 0)))


def verify_markov(U, E, W, anchor, draft_lse, draft_tok_logit, tgt_logits, tgt_off, ell, draft_tok, temperature,
                  seed: int, *, out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                  status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Verification with the rejecting draft rows recomputed (C ABI dspark_verify_markov).

    U [B,K_max,V], E [V,rank] bf16 and W [rank,V] bf16 or a PackedProjection of it, anchor [B]
    int32 -- the draft's inputs -- and its draft_lse, draft_tok_logit [B,K_max] float32 outputs;
    the rest as for verify_ragged.  Returns n_acc [B] and out_tok [B,K_max+1] (int32).
    """
    _dev(U, "U", torch.bfloat16)
    B, K_max, V = U.shape
    rank = E.shape[1]
    _dev(E, "E", torch.bfloat16, (V, rank))
    flags = 0
    if isinstance(W, PackedProjection):
        if (W.rank, W.V) != (rank, V) or W.device != U.device:
            raise ValueError(f"packed projection of shape ({W.rank}, {W.V}) does not fit U/E")
        flags |= FLAG_W_PACKED
        W = W.data
    else:
        _dev(W, "W", torch.bfloat16, (rank, V))
    _dev(anchor, "anchor", torch.int32, (B,))
    _dev(draft_lse, "draft_lse", torch.float32, (B, K_max))
    _dev(draft_tok_logit, "draft_tok_logit", torch.float32, (B, K_max))
    _dev(tgt_logits, "tgt_logits", torch.bfloat16)
    if tgt_logits.dim() != 2 or tgt_logits.shape[1] != V:
        raise ValueError("tgt_logits must be [rows, V]")
    _dev(tgt_off, "tgt_off", torch.int32, (B + 1,))
    _dev(ell, "ell", torch.int32, (B,))
    _dev(draft_tok, "draft_tok", torch.int32, (B, K_max))
    _dev(temperature, "temperature", torch.float32, (B,))
    dev = U.device
    out = {} if out is None else out
    n_acc = out.get("n_acc") if out.get("n_acc") is not None else torch.empty(B, dtype=torch.int32, device=dev)
    out_tok = out.get("out_tok") if out.get("out_tok") is not None else torch.empty(B, K_max + 1, dtype=torch.int32,
                                                                                    device=dev)
    status = new_status(dev) if status is None else status
    dims = Dims(B, K_max, V, rank, BF16, flags)
    nbytes = int(lib().dspark_verify_markov_workspace_bytes(dims))
    if nbytes == 0:
        _raise(13, "dspark_verify_markov")
    ws = _workspace(nbytes, dev, workspace)
    code = lib().dspark_verify_markov(_ptr(U), _ptr(E), _ptr(W), _ptr(anchor), _ptr(draft_lse), _ptr(draft_tok_logit),
                                      _ptr(tgt_logits), _ptr(tgt_off), _ptr(ell), _ptr(draft_tok), _ptr(temperature),
                                      ctypes.c_uint64(seed), dims, _ptr(n_acc), _ptr(out_tok), _ptr(ws),
                                      ctypes.c_size_t(ws.numel()), _ptr(status), _stream(stream))
    _raise(code, "dspark_verify_markov")
    return dict(n_acc=n_acc, out_tok=out_tok, status=status, workspace=ws)
