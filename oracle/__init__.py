"""CPU oracle for the DSpark per-step hot path (TEST INFRASTRUCTURE ONLY).

This package wraps ``dspark_oracle.c``: a plain, slow, fp64 statement of the
three hot-path operations (Markov-head draft sampling, survival scheduling,
ragged rejection-sampling verification) and of the Philox4x32-10 random stream
both implementations reproduce.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with
the CUDA library in ``speculative_decoding_draft_gb300``.

Sources: "DSpark: Confidence-Scheduled Speculative Decoding with
Semi-Autoregressive Generation" (S2.1, S3.1, S3.2.2 Algorithm 1, Appendix A);
"Speculative decoding, from zero to DSpark" (S2, S6, S8, Appendix A1);
Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11, S4).

Parity status: every exported function is pinned by tests/test_oracle_*.py
against worked numbers printed on the pages, closed forms, exhaustive search,
exact enumeration or published known-answer vectors.  No function is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_LIB = os.path.join(_HERE, "libdspark_oracle.so")

# Status names, oracle numbering (the CUDA library has its own enum; tests map by name).
STATUS = {
    0: "OK",
    1: "ERR_NULL",
    2: "ERR_DIMS",
    3: "ERR_DTYPE",
    4: "ERR_TEMPERATURE",
    5: "ERR_SPS_TOO_SHORT",
    6: "ERR_OFFSETS",
    7: "ERR_TOKEN_RANGE",
    8: "ERR_LENGTHS",
    9: "ERR_CONFIDENCE",
}

F32, BF16 = 0, 1
TAG_DRAFT, TAG_ACCEPT, TAG_RESID, TAG_DRAFT_PICK, TAG_RESID_PICK = 0, 1, 2, 3, 4


class OracleError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        self.name = STATUS.get(code, f"UNKNOWN({code})")
        super().__init__(f"oracle returned {self.name}")


def build(force: bool = False, openmp: bool = True) -> str:
    """Compile the oracle shared library in place (gcc, C11, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-D_DEFAULT_SOURCE"]
    tmp = _LIB + f".tmp{os.getpid()}"
    cmds = ([base + ["-fopenmp", "-o", tmp, _SRC, "-lm"]] if openmp else []) + [base + ["-o", tmp, _SRC, "-lm"]]
    last = None
    for cmd in cmds:
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _LIB)
            return _LIB
        last = r.stderr
    raise RuntimeError(f"oracle build failed:\n{last}")


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, u64, u32, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        L.dso_philox4x32_10.argtypes = [P, P, P]
        L.dso_philox4x32_10.restype = None
        L.dso_stream_word.argtypes = [u64, u64, u32, u32, u32]
        L.dso_stream_word.restype = u32
        for name in ("dso_uniform_open", "dso_uniform_accept", "dso_gumbel"):
            getattr(L, name).argtypes = [u32]
            getattr(L, name).restype = ctypes.c_double
        L.dso_round_bf16.argtypes = [ctypes.c_double]
        L.dso_round_bf16.restype = ctypes.c_double
        L.dso_draft_markov_sample.argtypes = [P, P, P, i32, P, P, P, P, u64, i64, i64, i64, i64,
                                              P, P, P, P, P, P, i32]
        L.dso_draft_markov_sample.restype = i32
        L.dso_draft_rnn_sample.argtypes = [P, P, P, P, i32, P, P, P, P, P, u64, i64, i64, i64, i64,
                                           P, P, P, P, P, P, P, i32]
        L.dso_draft_rnn_sample.restype = i32
        L.dso_schedule_survival.argtypes = [P, P, P, i64, i64, i64, P, P, P, P, P, P, P, P, P, P]
        L.dso_schedule_survival.restype = i32
        L.dso_draft_confidence.argtypes = [P, i32, i64, i64, P, P, P, P, P, i64, i64, P]
        L.dso_draft_confidence.restype = i32
        L.dso_schedule_capacity.argtypes = [P, P, P, i64, i64, i64, P, P, P, P, P]
        L.dso_schedule_capacity.restype = i32
        L.dso_schedule_topk.argtypes = [P, P, i64, i64, i64, P, P, P, P, P, P]
        L.dso_schedule_topk.restype = i32
        L.dso_schedule_threshold.argtypes = [P, P, i64, i64, ctypes.c_float, i32, P, P, P]
        L.dso_schedule_threshold.restype = i32
        L.dso_verify_ragged.argtypes = [P, P, i32, P, P, P, P, P, u64, i64, i64, i64,
                                        P, P, P, P, P, P, i32]
        L.dso_verify_ragged.restype = i32
        L.dso_row_lse.argtypes = [P, i32, i64, i64, P, P]
        L.dso_row_lse.restype = i32
        L.dso_block_race.argtypes = [P, P, i64, u64, u32, u32, u32, u32, P, P, P, P]
        L.dso_block_race.restype = i64
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# array marshalling
# ---------------------------------------------------------------------------
def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _logits(a):
    """Accept float32 arrays, or bf16 given as uint16 bit patterns; return (array, dtype code)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _threads(nthreads):
    return int(nthreads) if nthreads else 0


# ---------------------------------------------------------------------------
# random stream
# ---------------------------------------------------------------------------
def philox4x32_10(counter, key):
    ctr = _c(counter, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().dso_philox4x32_10(_ptr(ctr), _ptr(k), _ptr(out))
    return out


def stream_word(seed, v, position, request, tag):
    return int(lib().dso_stream_word(int(seed), int(v), int(position), int(request), int(tag)))


def uniform_open(w):
    return float(lib().dso_uniform_open(int(w)))


def uniform_accept(w):
    return float(lib().dso_uniform_accept(int(w)))


def gumbel(w):
    return float(lib().dso_gumbel(int(w)))


def round_bf16(x):
    return float(lib().dso_round_bf16(float(x)))


def block_race(log_w, seed, position, request, tag_block, tag_pick, log_err=None):
    """Two-level categorical draw over weights exp(log_w) (-inf = zero weight).

    Returns dict(pick, block, score, margin, near_block, near_pick, near_err).
    """
    lw = _c(log_w, np.float64)
    le = None if log_err is None else _c(log_err, np.float64)
    blk = ctypes.c_int64(0)
    score = ctypes.c_double(0)
    margin = ctypes.c_double(0)
    near = np.zeros(3, np.int32)
    pick = lib().dso_block_race(_ptr(lw), _ptr(le), lw.size, int(seed), int(position), int(request),
                                int(tag_block), int(tag_pick), ctypes.byref(blk), ctypes.byref(score),
                                ctypes.byref(margin), _ptr(near))
    return dict(pick=int(pick), block=int(blk.value), score=score.value, margin=margin.value,
                near_block=bool(near[0]), near_pick=bool(near[1]), near_err=bool(near[2]))


# ---------------------------------------------------------------------------
# hot-path operations
# ---------------------------------------------------------------------------
def draft_markov_sample(U, E, W, anchor, K_r, temperature, seed, req_id=None, want_logits=True,
                        want_spread=False, nthreads=0):
    """Markov-head draft sampling.  U: [B, K_max, V]; E: [V, rank]; W: [rank, V].

    Returns dict(draft_tok [B,K_max] int32, draft_logits (same dtype as U) or None,
    lse [B,K_max] f64, margin [B,K_max] f64, flags [B,K_max] u8, spread).  With want_spread
    (bf16), spread [B,K_max,V] f32 bounds, per stored logit, how far another fp32 evaluation
    of U + bias may move it: 0 where none can change it, one bf16 step where the exact value
    sits within the fp32 error bound of a rounding midpoint, more where the sum cancels to
    near zero; else None.
    """
    U, dt = _logits(U)
    E, dtE = _logits(E)
    W, dtW = _logits(W)
    if not (dt == dtE == dtW):
        raise TypeError("U, E, W must share one dtype")
    B, K_max, V = U.shape
    rank = E.shape[1]
    if E.shape[0] != V or W.shape != (rank, V):
        raise ValueError("shape mismatch")
    anchor = _c(anchor, np.int32)
    K_r = _c(K_r, np.int32)
    temperature = _c(temperature, np.float32)
    rid = None if req_id is None else _c(req_id, np.int64)
    tok = np.zeros((B, K_max), np.int32)
    logits = np.zeros_like(U) if want_logits else None
    lse = np.zeros((B, K_max), np.float64)
    margin = np.zeros((B, K_max), np.float64)
    flags = np.zeros((B, K_max), np.uint8)
    spread = np.zeros((B, K_max, V), np.float32) if want_spread else None
    st = lib().dso_draft_markov_sample(_ptr(U), _ptr(E), _ptr(W), dt, _ptr(anchor), _ptr(K_r),
                                       _ptr(temperature), _ptr(rid), int(seed), B, K_max, V, rank,
                                       _ptr(tok), _ptr(logits), _ptr(lse), _ptr(margin), _ptr(flags),
                                       _ptr(spread), _threads(nthreads))
    if st:
        raise OracleError(st)
    return dict(draft_tok=tok, draft_logits=logits, lse=lse, margin=margin, flags=flags, spread=spread)


def draft_rnn_sample(U, E, W, Wc, cx, anchor, K_r, temperature, seed, req_id=None, want_logits=True,
                     want_feat=False, want_spread=False, nthreads=0):
    """RNN-head draft sampling.  U [B,K_max,V]; E [V,rank]; W [rank,V]; Wc [3 rank, 2 rank] (one dtype);
    cx [B,K_max,3 rank] float32 (the backbone term of the cell).

    Returns the draft_markov_sample dict plus feat [B,K_max,rank] f64 (the head's feature) when asked.
    The spread's error bound adds the feature's own fp32 error (at most 1e-5 per component) to
    the Markov head's summation bound.
    """
    U, dt = _logits(U)
    E, dtE = _logits(E)
    W, dtW = _logits(W)
    Wc, dtC = _logits(Wc)
    if not (dt == dtE == dtW == dtC):
        raise TypeError("U, E, W, Wc must share one dtype")
    B, K_max, V = U.shape
    rank = E.shape[1]
    if E.shape[0] != V or W.shape != (rank, V) or Wc.shape != (3 * rank, 2 * rank):
        raise ValueError("shape mismatch")
    cx = _c(cx, np.float32)
    if cx.shape != (B, K_max, 3 * rank):
        raise ValueError("cx shape mismatch")
    anchor = _c(anchor, np.int32)
    K_r = _c(K_r, np.int32)
    temperature = _c(temperature, np.float32)
    rid = None if req_id is None else _c(req_id, np.int64)
    tok = np.zeros((B, K_max), np.int32)
    logits = np.zeros_like(U) if want_logits else None
    lse = np.zeros((B, K_max), np.float64)
    margin = np.zeros((B, K_max), np.float64)
    flags = np.zeros((B, K_max), np.uint8)
    feat = np.zeros((B, K_max, rank), np.float64) if want_feat else None
    spread = np.zeros((B, K_max, V), np.float32) if want_spread else None
    st = lib().dso_draft_rnn_sample(_ptr(U), _ptr(E), _ptr(W), _ptr(Wc), dt, _ptr(cx), _ptr(anchor), _ptr(K_r),
                                    _ptr(temperature), _ptr(rid), int(seed), B, K_max, V, rank, _ptr(tok),
                                    _ptr(logits), _ptr(lse), _ptr(margin), _ptr(flags), _ptr(feat), _ptr(spread),
                                    _threads(nthreads))
    if st:
        raise OracleError(st)
    return dict(draft_tok=tok, draft_logits=logits, lse=lse, margin=margin, flags=flags, feat=feat, spread=spread)


def draft_confidence(E, anchor, draft_tok, K_r, conf_h, conf_w):
    """Confidence head with the Markov term: c_k = sigmoid(conf_h[r, k] + conf_w . E[x_{k-1}]).

    E [V, rank] float32 or bf16 bits (uint16); draft_tok [B, K_max] int32 (x_1..); conf_h
    [B, K_max] float32 (w_h . h_k + b); conf_w [rank] float32.  Returns conf [B, K_max] float32.
    """
    Ea, dt = _logits(E)
    V, rank = Ea.shape
    draft_tok = _c(draft_tok, np.int32)
    B, K_max = draft_tok.shape
    anchor = _c(anchor, np.int32)
    K_r = _c(K_r, np.int32)
    conf_h = _c(conf_h, np.float32)
    conf_w = _c(conf_w, np.float32)
    out = np.zeros((B, K_max), np.float32)
    st = lib().dso_draft_confidence(_ptr(Ea), dt, V, rank, _ptr(anchor), _ptr(draft_tok), _ptr(K_r), _ptr(conf_h),
                                    _ptr(conf_w), B, K_max, _ptr(out))
    if st:
        raise OracleError(st)
    return out


def schedule_survival(conf, K_r, sps):
    """Hardware-aware prefix scheduler (Algorithm 1).  conf: [B, K_max] f32; sps: f64 table."""
    conf = _c(conf, np.float32)
    B, K_max = conf.shape
    K_r = _c(K_r, np.int32)
    sps = _c(sps, np.float64)
    ell = np.zeros(B, np.int32)
    off = np.zeros(B + 1, np.int32)
    th = np.zeros(1, np.float64)
    bstar = np.zeros(1, np.int64)
    tau = np.zeros(1, np.float64)
    surv = np.zeros((B, K_max), np.float32)
    order = np.zeros(B * K_max, np.int32)
    ncand = np.zeros(1, np.int64)
    nadm = np.zeros(1, np.int64)
    ties = np.zeros(1, np.int64)
    st = lib().dso_schedule_survival(_ptr(conf), _ptr(K_r), _ptr(sps), len(sps), B, K_max,
                                     _ptr(ell), _ptr(off), _ptr(th), _ptr(bstar), _ptr(tau),
                                     _ptr(surv), _ptr(order), _ptr(ncand), _ptr(nadm), _ptr(ties))
    if st:
        raise OracleError(st)
    n = int(ncand[0])
    return dict(ell=ell, tgt_off=off, theta_best=float(th[0]), B_star=int(bstar[0]),
                tau_star=float(tau[0]), survival=surv, order=order[:n], n_cand=n,
                n_admitted=int(nadm[0]), n_theta_ties=int(ties[0]))


def schedule_capacity(conf, K_r, sps):
    """Capacity of the asynchronous scheduler: the global maximum of Theta along the greedy path.

    Returns dict(capacity, theta_best, ell, tgt_off, survival); ell is the admission at the maximum.
    """
    conf = _c(conf, np.float32)
    B, K_max = conf.shape
    K_r = _c(K_r, np.int32)
    sps = _c(sps, np.float64)
    cap = np.zeros(1, np.int64)
    th = np.zeros(1, np.float64)
    ell = np.zeros(B, np.int32)
    off = np.zeros(B + 1, np.int32)
    surv = np.zeros((B, K_max), np.float32)
    st = lib().dso_schedule_capacity(_ptr(conf), _ptr(K_r), _ptr(sps), len(sps), B, K_max, _ptr(cap), _ptr(th),
                                     _ptr(ell), _ptr(off), _ptr(surv))
    if st:
        raise OracleError(st)
    return dict(capacity=int(cap[0]), theta_best=float(th[0]), ell=ell, tgt_off=off, survival=surv)


def schedule_topk(conf, K_r, capacity):
    """Dynamic top-K admission: the first min(capacity, N) candidates of the current ranking."""
    conf = _c(conf, np.float32)
    B, K_max = conf.shape
    K_r = _c(K_r, np.int32)
    ell = np.zeros(B, np.int32)
    off = np.zeros(B + 1, np.int32)
    nadm = np.zeros(1, np.int64)
    surv = np.zeros((B, K_max), np.float32)
    order = np.zeros(B * K_max, np.int32)
    ncand = np.zeros(1, np.int64)
    st = lib().dso_schedule_topk(_ptr(conf), _ptr(K_r), B, K_max, int(capacity), _ptr(ell), _ptr(off), _ptr(nadm),
                                 _ptr(surv), _ptr(order), _ptr(ncand))
    if st:
        raise OracleError(st)
    n = int(ncand[0])
    return dict(ell=ell, tgt_off=off, n_admitted=int(nadm[0]), survival=surv, order=order[:n], n_cand=n)


THRESHOLD_CONFIDENCE, THRESHOLD_SURVIVAL = 0, 1


def schedule_threshold(conf, K_r, theta, mode=THRESHOLD_CONFIDENCE):
    """Static-threshold lengths: the longest prefix whose confidences (mode 0) or survivals (mode 1) are >= theta."""
    conf = _c(conf, np.float32)
    B, K_max = conf.shape
    K_r = _c(K_r, np.int32)
    ell = np.zeros(B, np.int32)
    off = np.zeros(B + 1, np.int32)
    surv = np.zeros((B, K_max), np.float32)
    st = lib().dso_schedule_threshold(_ptr(conf), _ptr(K_r), B, K_max, float(theta), int(mode), _ptr(ell),
                                      _ptr(off), _ptr(surv))
    if st:
        raise OracleError(st)
    return dict(ell=ell, tgt_off=off, survival=surv)


def verify_ragged(draft_logits, tgt_logits, tgt_off, ell, draft_tok, temperature, seed, req_id=None,
                  draft_spread=None, nthreads=0):
    """Ragged rejection-sampling verification.

    draft_logits [B, K_max, V]; tgt_logits [sum(ell+1), V] flattened; tgt_off [B+1].
    draft_spread (optional) [B, K_max, V] f32: the draft's spreads (draft_markov_sample's
    spread); decisions that another fp32 evaluation of the draft logits could move are
    flagged.
    Returns dict(n_acc [B], out_tok [B, K_max+1], flags [B], flag_pos [B], sample_margin [B]).
    """
    D, dt = _logits(draft_logits)
    Tg, dt2 = _logits(tgt_logits)
    if dt != dt2:
        raise TypeError("draft and target logits must share one dtype")
    B, K_max, V = D.shape
    tgt_off = _c(tgt_off, np.int32)
    ell = _c(ell, np.int32)
    draft_tok = _c(draft_tok, np.int32)
    temperature = _c(temperature, np.float32)
    rid = None if req_id is None else _c(req_id, np.int64)
    n_acc = np.zeros(B, np.int32)
    out = np.zeros((B, K_max + 1), np.int32)
    flags = np.zeros(B, np.uint8)
    fpos = np.zeros(B, np.int32)
    mg = np.zeros(B, np.float64)
    amb = None
    if draft_spread is not None:
        amb = _c(draft_spread, np.float32)
        if amb.shape != D.shape:
            raise ValueError("draft_spread must have the draft logits' shape")
    st = lib().dso_verify_ragged(_ptr(D), _ptr(Tg), dt, _ptr(tgt_off), _ptr(ell), _ptr(draft_tok),
                                 _ptr(temperature), _ptr(rid), int(seed), B, K_max, V, _ptr(amb),
                                 _ptr(n_acc), _ptr(out), _ptr(flags), _ptr(fpos), _ptr(mg),
                                 _threads(nthreads))
    if st:
        raise OracleError(st)
    return dict(n_acc=n_acc, out_tok=out, flags=flags, flag_pos=fpos, sample_margin=mg)


def row_lse(rows, row_temperature):
    """fp64 log-sum-exp of each row of z/T (row max when T = 0)."""
    R, dt = _logits(rows)
    V = R.shape[-1]
    R2 = R.reshape(-1, V)
    t = _c(row_temperature, np.float32).reshape(-1)
    out = np.zeros(R2.shape[0], np.float64)
    st = lib().dso_row_lse(_ptr(R2), dt, R2.shape[0], V, _ptr(t), _ptr(out))
    if st:
        raise OracleError(st)
    return out.reshape(R.shape[:-1])


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
