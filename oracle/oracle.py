"""ctypes wrapper around the plain-C fp64 oracle (kvev_oracle.c).

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU leg).  The wrapper
marshals numpy arrays; every step of the method is computed in the C file.

Refresh schedule, "What Matters for Aggressive Decoding-Time KV Eviction?"
Sec. 3.2: full refresh scores every step; lazy refresh with period r scores at
steps t with (t-1) mod r == 0 (Eq. 6); Score-Free scores at step 1 only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvev_oracle.c")
_LIB = os.path.join(_HERE, "libkvev_oracle.so")
_lib = None

REFRESH_FULL, REFRESH_LAZY, REFRESH_FROZEN = 0, 1, 2
AGG_EMA, AGG_CUMULATIVE = 0, 1
W_VNORM, W_ENTROPY = 1, 2
AGE_SINCE_INSERT, AGE_SINCE_ACCESS = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain IEEE fp64: no fast-math, no FMA
    contraction).  Returns the shared-library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-fopenmp", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.kvo_ema.restype = ctypes.c_double
        lib.kvo_ema.argtypes = [ctypes.c_double] * 3
        lib.kvo_priority.restype = ctypes.c_double
        lib.kvo_priority.argtypes = [ctypes.c_double, ctypes.c_int64, ctypes.c_double]
        lib.kvo_attention.restype = None
        lib.kvo_attention.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                      P, P, P, ctypes.c_int64, P, P]
        lib.kvo_select.restype = ctypes.c_int64
        lib.kvo_select.argtypes = [ctypes.c_int64, P, P, ctypes.c_int64, P]
        lib.kvo_set_threads.restype = ctypes.c_int
        lib.kvo_set_threads.argtypes = [ctypes.c_int]
        lib.kvo_step.restype = ctypes.c_int64
        lib.kvo_step.argtypes = ([P, ctypes.c_int64, ctypes.c_int, ctypes.c_int64]
                                 + [P] * 6 + [ctypes.c_int64] + [P] * 17)
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class _Params(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cap", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
                ("budget", ctypes.c_int64), ("alpha", ctypes.c_double),
                ("beta", ctypes.c_double), ("age_mode", ctypes.c_int32),
                ("pool_mean", ctypes.c_int32), ("aggregation", ctypes.c_int32),
                ("weighting", ctypes.c_int32)]


def set_threads(n: int = 0) -> int:
    """Host threads of the attention (n >= 1; 0 keeps the current count).
    Returns the count in effect.  Results do not depend on it."""
    return int(_load().kvo_set_threads(int(n)))


# ------------------------------------------------------------- scalar rules
def ema(score: float, new_score: float, alpha: float) -> float:
    return _load().kvo_ema(score, new_score, alpha)


def priority(score: float, steps: int, beta: float) -> float:
    return _load().kvo_priority(score, int(steps), beta)


def is_refresh(mode: int, period: int, t: int) -> bool:
    if mode == REFRESH_FULL:
        return True
    if mode == REFRESH_LAZY:
        return (t - 1) % period == 0
    if mode == REFRESH_FROZEN:
        return t == 1
    raise ValueError(mode)


def select(pr, budget: int, pinned=None) -> np.ndarray:
    pr = np.ascontiguousarray(pr, dtype=np.float64)
    L = pr.shape[0]
    pin = None if pinned is None else np.ascontiguousarray(pinned, dtype=np.uint8)
    kept = np.zeros(max(L, 1), dtype=np.int64)
    n = _load().kvo_select(L, _ptr(pr), _ptr(pin), int(budget), _ptr(kept))
    return kept[:n].copy()


def attention(q_bits, k_bits, v_bits):
    """q [Hq][d], k/v [Hkv][L][d] bf16 bits -> (probs [Hq][L], out [Hq][d])."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    Hq, d = q.shape
    Hkv, L, _ = k.shape
    probs = np.zeros((Hq, L), dtype=np.float64)
    out = np.zeros((Hq, d), dtype=np.float64)
    _load().kvo_attention(Hq, Hkv, d, L, _ptr(q), _ptr(k), _ptr(v), L, _ptr(probs), _ptr(out))
    return probs, out


# ------------------------------------------------------------------ stepping
@dataclass
class OracleParams:
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    budget: int
    alpha: float
    beta: float
    age_mode: int = AGE_SINCE_INSERT
    pool_mean: bool = False
    aggregation: int = 0      # AGG_EMA or AGG_CUMULATIVE (p1 Sec. 3.1 Eqs. (3), (4))
    weighting: int = 0        # W_VNORM | W_ENTROPY (p1 Appendix E "Per-step scoring")


@dataclass
class SequenceState:
    """Host copy of one sequence's cache and per-token state.

    K, V: uint16 [Ly][Hkv][cap][d]; m float64 [cap]; t_ins, t_ref, pos int64
    [cap]; L = number of live slots."""
    K: np.ndarray
    V: np.ndarray
    m: np.ndarray
    t_ins: np.ndarray
    t_ref: np.ndarray
    pos: np.ndarray
    L: int
    extra: dict = field(default_factory=dict)

    @staticmethod
    def from_prefill(K, V, L0: int, cap: int) -> "SequenceState":
        """K, V: [Ly][Hkv][L0][d] bits; all prefill tokens inserted at step 0."""
        Ly, Hkv, _, d = K.shape
        Kc = np.zeros((Ly, Hkv, cap, d), dtype=np.uint16)
        Vc = np.zeros((Ly, Hkv, cap, d), dtype=np.uint16)
        Kc[:, :, :L0] = K
        Vc[:, :, :L0] = V
        z = np.zeros(cap, dtype=np.int64)
        pos = z.copy()
        pos[:L0] = np.arange(L0)
        return SequenceState(Kc, Vc, np.zeros(cap), z.copy(), z.copy(), pos, L0)

    def copy(self) -> "SequenceState":
        return SequenceState(self.K.copy(), self.V.copy(), self.m.copy(), self.t_ins.copy(),
                             self.t_ref.copy(), self.pos.copy(), self.L, dict(self.extra))


def step(P: OracleParams, st: SequenceState, t: int, refresh: bool, q_bits, knew_bits,
         vnew_bits, new_pos: int, forced_access=None, want_probs: bool = True):
    """One decode step of one sequence.  Returns (result dict, new state); the
    input state is not modified.  q [Ly][Hq][d], k_new/v_new [Ly][Hkv][d]."""
    lib = _load()
    Ly, Hkv, cap, d = st.K.shape
    if st.L + 1 > cap:
        raise ValueError("cache capacity exceeded")
    work = st.copy()
    L = st.L + 1
    prm = _Params(P.n_layers, P.n_q_heads, P.n_kv_heads, P.head_dim, cap, Hkv * cap * d,
                  P.budget, P.alpha, P.beta, P.age_mode, int(P.pool_mean),
                  int(P.aggregation), int(P.weighting))
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kn = np.ascontiguousarray(knew_bits, dtype=np.uint16)
    vn = np.ascontiguousarray(vnew_bits, dtype=np.uint16)
    fa = None if forced_access is None else np.ascontiguousarray(forced_access, dtype=np.int8)
    out = np.zeros((Ly, P.n_q_heads, d))
    probs = np.zeros((Ly, P.n_q_heads, L)) if want_probs else None
    ssum = np.zeros(L)
    m_upd = np.zeros(L)
    pr = np.zeros(L)
    acc = np.zeros(L, dtype=np.uint8)
    retained = np.zeros(L, dtype=np.int64)
    new = SequenceState(np.zeros_like(st.K), np.zeros_like(st.V), np.zeros(cap),
                        np.zeros(cap, np.int64), np.zeros(cap, np.int64),
                        np.zeros(cap, np.int64), 0)
    n = lib.kvo_step(ctypes.byref(prm), t, int(bool(refresh)), st.L, _ptr(work.K), _ptr(work.V),
                     _ptr(work.m), _ptr(work.t_ins), _ptr(work.t_ref), _ptr(work.pos),
                     int(new_pos), _ptr(q), _ptr(kn), _ptr(vn), _ptr(fa), _ptr(out),
                     _ptr(probs), _ptr(ssum), _ptr(m_upd), _ptr(pr), _ptr(acc),
                     _ptr(retained), _ptr(new.K), _ptr(new.V), _ptr(new.m),
                     _ptr(new.t_ins), _ptr(new.t_ref), _ptr(new.pos))
    new.L = int(n)
    res = dict(out=out, probs=probs, score_sum=ssum, m_upd=m_upd, priority=pr,
               accessed=acc.astype(bool), retained=retained[:n].copy(), L=L,
               t_ref_upd=work.t_ref[:L].copy())
    return res, new
