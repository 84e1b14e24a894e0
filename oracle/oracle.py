"""ctypes front end of the fp64 CPU oracle (``dspark_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers.  The CUDA library never imports this module, and this module
imports nothing from the CUDA library: inputs arrive as numpy arrays (bf16 as raw uint16 bit
patterns) and every result is computed in double precision by the C++ file next to it.

``build()`` compiles the oracle with the host C++ compiler (``g++ -O2 -fopenmp``); it is plain
portable C++ and builds the same way on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

DT_F32, DT_BF16, DT_F64 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or older than its source."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared",
           "-ffp-contract=off", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every call of this front end to another build of the oracle while the block runs.
    The planted-mistake tests compile mutated copies of ``dspark_oracle.cpp`` and check that the
    pins reject each one."""
    global _lib
    saved = _lib
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def _bind(lib):
    """Declare the argument and result types of the oracle's exported functions on ``lib``."""
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.orc_philox4x32_10.argtypes = [P, P, P]
    lib.orc_philox4x32_10.restype = None
    lib.orc_uniform.argtypes = [ctypes.c_uint64, I, I, ctypes.c_int64]
    lib.orc_uniform.restype = ctypes.c_double
    lib.orc_gumbel.argtypes = [ctypes.c_uint64, I, I, ctypes.c_int64]
    lib.orc_gumbel.restype = ctypes.c_double
    lib.orc_draft.argtypes = ([I, I, I, I, I, I, ctypes.c_double, ctypes.c_uint64, I,
                               P, P, P, I, P, P, P, P, P, P, P, P, I]
                              + [P] * 11 + [I])
    lib.orc_draft.restype = I
    lib.orc_confidence.argtypes = [I, I, I, I, I, I, P, I, P, P, P, P, P, P]
    lib.orc_confidence.restype = I
    lib.orc_tv_label.argtypes = [I, I, ctypes.c_double, P, P, P, P, I]
    lib.orc_tv_label.restype = None
    lib.orc_verify.argtypes = [I, I, I, ctypes.c_double, ctypes.c_uint64] + [P] * 9 + [I]
    lib.orc_verify.restype = I
    lib.orc_draft_loss.argtypes = ([I, I, I, ctypes.c_double, P, P, P, P] + [ctypes.c_double] * 3
                                   + [P] * 4 + [I])
    lib.orc_draft_loss.restype = I
    lib.orc_sts.argtypes = [I, I, P, P, I, P, I, P, P, P]
    lib.orc_sts.restype = I
    lib.orc_prefix_schedule.argtypes = [I, I, P, P, P, P]
    lib.orc_prefix_schedule.restype = I
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dt(a) -> int:
    if a.dtype == np.float32:
        return DT_F32
    if a.dtype == np.uint16:
        return DT_BF16
    if a.dtype == np.float64:
        return DT_F64
    raise TypeError(f"unsupported oracle dtype {a.dtype}")


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


def philox4x32_10(counter, key) -> np.ndarray:
    ctr = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_ptr(ctr), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, b: int, k: int, v: int) -> float:
    return _load().orc_uniform(seed, b, k, v)


def gumbel(seed: int, b: int, k: int, v: int) -> float:
    return _load().orc_gumbel(seed, b, k, v)


@dataclass
class DraftResult:
    tokens: np.ndarray   # [n, gamma] int32
    best: np.ndarray     # [n, gamma] winning perturbed score y + g
    tokens2: np.ndarray  # [n, gamma] runner-up token
    best2: np.ndarray    # [n, gamma] runner-up perturbed score
    lse: np.ndarray      # [n, gamma] log-sum-exp of y = z / T
    c: np.ndarray | None
    S: np.ndarray | None
    cstar: np.ndarray | None
    l1: np.ndarray | None
    z: np.ndarray | None      # [n, gamma, V] logits before temperature, when requested
    s_final: np.ndarray | None
    status: int


def draft(*, head: int, B: int, gamma: int, V: int, r: int, d: int, T: float, seed: int,
          W1, W2, U, x0, Wj=None, h=None, w=None, target=None, s0=None, forced=None,
          rows=None, want_z: bool = False, nthreads: int = 0) -> DraftResult:
    """Run the oracle draft for the requests in ``rows`` (all requests when None).

    Weight arrays (W1, W2, Wj, w) share one dtype and activations (U, h) another; fp32 arrays
    are float32, bf16 arrays are the raw uint16 patterns.  ``target`` is float32.
    """
    W1, W2, Wj, w = _c(W1), _c(W2), _c(Wj), _c(w)
    U, h = _c(U), _c(h)
    wdt, udt = _dt(W1), _dt(U)
    for a in (W2, Wj, w):
        if a is not None and _dt(a) != wdt:
            raise TypeError("weights must share one dtype")
    if h is not None and _dt(h) != udt:
        raise TypeError("h must share U's dtype")
    x0 = _c(x0, np.int32)
    target = _c(target, np.float32)
    s0 = _c(s0, np.float64)
    forced = _c(forced, np.int32)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = B if rows_a is None else len(rows_a)
    f = lambda dt: np.zeros((n, gamma), dtype=dt)
    tok, tok2 = f(np.int32), f(np.int32)
    best, best2, lse = f(np.float64), f(np.float64), f(np.float64)
    conf = h is not None and w is not None
    c = f(np.float64) if conf else None
    S = f(np.float64) if conf else None
    cstar = f(np.float64) if target is not None else None
    l1 = f(np.float64) if target is not None else None
    z = np.zeros((n, gamma, V), dtype=np.float64) if want_z else None
    s_out = np.zeros((n, r), dtype=np.float64) if head == 1 else None
    st = _load().orc_draft(
        head, B, gamma, V, r, d, float(T), seed, wdt, _ptr(W1), _ptr(W2), _ptr(Wj), udt,
        _ptr(U), _ptr(x0), _ptr(h), _ptr(w), _ptr(target), _ptr(s0), _ptr(forced),
        _ptr(rows_a), n, _ptr(tok), _ptr(best), _ptr(tok2), _ptr(best2), _ptr(lse), _ptr(c),
        _ptr(S), _ptr(cstar), _ptr(l1), _ptr(z), _ptr(s_out), nthreads)
    return DraftResult(tok, best, tok2, best2, lse, c, S, cstar, l1, z, s_out, st)


def confidence(*, B, gamma, V, r, d, W1, h, w, x0, tokens):
    W1, h, w = _c(W1), _c(h), _c(w)
    x0, tokens = _c(x0, np.int32), _c(tokens, np.int32)
    c = np.zeros((B, gamma), dtype=np.float64)
    S = np.zeros((B, gamma), dtype=np.float64)
    st = _load().orc_confidence(B, gamma, V, r, d, _dt(W1), _ptr(W1), _dt(h), _ptr(h), _ptr(w),
                                _ptr(x0), _ptr(tokens), _ptr(c), _ptr(S))
    return c, S, st


def tv_label(draft_logits, target_logits, T: float = 1.0, nthreads: int = 0):
    d = _c(draft_logits, np.float32)
    t = _c(target_logits, np.float32)
    N, V = d.shape
    cstar = np.zeros(N, dtype=np.float64)
    l1 = np.zeros(N, dtype=np.float64)
    _load().orc_tv_label(N, V, float(T), _ptr(d), _ptr(t), _ptr(cstar), _ptr(l1), nthreads)
    return cstar, l1


def prefix_schedule(S, sps):
    S = _c(S, np.float32)
    sps = _c(sps, np.float64)
    B, gamma = S.shape
    if sps.shape[0] < B * (gamma + 1) + 1:
        raise ValueError("sps needs B*(gamma+1)+1 entries")
    ln = np.zeros(B, dtype=np.int32)
    theta = np.zeros(1, dtype=np.float64)
    st = _load().orc_prefix_schedule(B, gamma, _ptr(S), _ptr(sps), _ptr(ln), _ptr(theta))
    return ln, float(theta[0]), st


@dataclass
class VerifyResult:
    n_accepted: np.ndarray  # [B] int32, -1 for a request with an invalid drafted token
    tokens: np.ndarray      # [B, gamma + 1] accepted prefix, then the correction or bonus; -1 after
    margin: np.ndarray      # [B, gamma] (ln q - ln p)(x_j) - ln a_j where tested, NaN after
    best: np.ndarray        # [B] winning perturbed score of the correction / bonus draw
    best2: np.ndarray       # [B] runner-up score
    tokens2: np.ndarray     # [B] runner-up id
    status: int


def verify(*, gamma: int, T: float, seed: int, draft_logits, target_logits, draft_tokens,
           nthreads: int = 0) -> VerifyResult:
    """The speculative accept/reject rule on one draft block per request.

    ``draft_logits`` is float32 [B, gamma, V], ``target_logits`` float32 [B, gamma + 1, V],
    ``draft_tokens`` int32 [B, gamma].
    """
    zd = _c(draft_logits, np.float32)
    zt = _c(target_logits, np.float32)
    x = _c(draft_tokens, np.int32)
    B, g, V = zd.shape
    if g != gamma or zt.shape != (B, gamma + 1, V) or x.shape != (B, gamma):
        raise ValueError("shapes: draft [B, gamma, V], target [B, gamma + 1, V], tokens [B, gamma]")
    n = np.zeros(B, dtype=np.int32)
    out = np.zeros((B, gamma + 1), dtype=np.int32)
    margin = np.zeros((B, gamma), dtype=np.float64)
    best = np.zeros(B, dtype=np.float64)
    best2 = np.zeros(B, dtype=np.float64)
    tok2 = np.zeros(B, dtype=np.int32)
    st = _load().orc_verify(B, gamma, V, float(T), seed, _ptr(zd), _ptr(zt), _ptr(x), _ptr(n),
                            _ptr(out), _ptr(margin), _ptr(best), _ptr(best2), _ptr(tok2), nthreads)
    return VerifyResult(n, out, margin, best, best2, tok2, st)


@dataclass
class LossResult:
    loss: np.ndarray         # [B] L = a_ce L_ce + a_tv L_tv + a_conf L_conf
    parts: np.ndarray        # [B, 3] (L_ce, L_tv, L_conf)
    grad_logits: np.ndarray  # [B, gamma, V] dL / d draft logits
    grad_conf: np.ndarray    # [B, gamma] dL / d confidence logits
    status: int


def draft_loss(*, T: float, draft_logits, target_logits, labels, conf_logits,
               alpha=(0.1, 0.9, 1.0), nthreads: int = 0) -> LossResult:
    """Eqs 9-12 and their gradients for draft logits [B, gamma, V] fp32, frozen target logits
    [B, gamma, V] fp32, labels [B, gamma] int32 and confidence logits [B, gamma] fp32."""
    zd = _c(draft_logits, np.float32)
    zt = _c(target_logits, np.float32)
    lab = _c(labels, np.int32)
    cf = _c(conf_logits, np.float32)
    B, gamma, V = zd.shape
    loss = np.zeros(B)
    parts = np.zeros((B, 3))
    gz = np.zeros((B, gamma, V))
    gc = np.zeros((B, gamma))
    st = _load().orc_draft_loss(B, gamma, V, float(T), _ptr(zd), _ptr(zt), _ptr(lab), _ptr(cf),
                                float(alpha[0]), float(alpha[1]), float(alpha[2]), _ptr(loss),
                                _ptr(parts), _ptr(gz), _ptr(gc), nthreads)
    return LossResult(loss, parts, gz, gc, st)


def sts(conf_logits, accepted, grid, bins: int = 15):
    """Sequential temperature scaling: per-position temperatures from the grid minimising the
    ECE of the cumulative product, left to right.  Returns (tau [gamma], ece [gamma],
    ece_grid [gamma, len(grid)], status)."""
    cf = _c(conf_logits, np.float32)
    acc = _c(accepted, np.int32)
    gr = _c(grid, np.float32)
    N, gamma = cf.shape
    tau = np.zeros(gamma)
    ece = np.zeros(gamma)
    eg = np.zeros((gamma, len(gr)))
    st = _load().orc_sts(N, gamma, _ptr(cf), _ptr(acc), len(gr), _ptr(gr), bins, _ptr(tau),
                         _ptr(ece), _ptr(eg))
    return tau, ece, eg, st
