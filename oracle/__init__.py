"""Plain CPU oracle for the speculative-decoding target-verification round.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The product library
never does, and this package imports nothing from the product.

The arithmetic lives in ``spec_oracle.c`` (fp64 accumulation, sequential
accept loop); this module compiles it with gcc and wraps it with numpy.
``exact_v16.py`` holds the exact-rational lossless check at V=16.

Readings of the pages that the oracle encodes (each one is also listed in the
design notes):
  * canonical Q4/Q6/Q8 block layout (the pages name Q4/Q6 and q8_0/q4_0
    block formats but do not fix a bit layout);
  * RMSNorm eps, rotate-half RoPE with theta, fp32 residual stream;
  * argmax ties go to the lowest index;
  * the strict rejection sampler's probabilities are integer weights
    ``floor(exp_own(z - max z) * 2^32)``, so that every decision is an exact
    integer comparison;
  * Philox4x32-10 counter = (slot lo, slot hi, sequence id, domain),
    key = (seed lo, seed hi); pinned against cuRAND's host-side Philox
    generator (counter words 0-2, key schedule; word 3 only at 0).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
             "-shared", "-fPIC", "-std=gnu11"]


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into oracle/_build/liboracle.so (gcc)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int
U64 = ctypes.c_uint64
U32 = ctypes.c_uint32
F32 = ctypes.c_float
F64 = ctypes.c_double


class _QW(ctypes.Structure):
    _fields_ = [("qtype", ctypes.c_int), ("qs", P), ("qh", P), ("scales", P),
                ("N", I64), ("K", I64)]


class _Desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("max_ctx", I64), ("rms_eps", F64),
                ("rope_theta", F64), ("use_rope", ctypes.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            sig = {
                "oracle_f64_to_f16": (None, [P, I64, P]),
                "oracle_f16_to_f64": (None, [P, I64, P]),
                "oracle_dequant": (None, [I32, P, P, P, I64, I64, I64, I64, P]),
                "oracle_linear": (None, [I32, P, P, P, I64, I64, P, I64, P]),
                "oracle_rmsnorm": (None, [P, P, I64, I64, F64, P]),
                "oracle_rope": (None, [P, I64, I32, P, F64, P]),
                "oracle_attention": (None, [P, I64, I32, I32, I32, P, P, I64, P, P]),
                "oracle_swiglu": (None, [P, P, I64, P]),
                "oracle_forward": (None, [P, P, P, P, P, P, P, P, I32, I32, P, P,
                                          P, P, P]),
                "oracle_argmax": (I64, [P, I64]),
                "oracle_accept_greedy": (I32, [P, P, I32, I32, P, P]),
                "oracle_exp_own": (F32, [F32]),
                "oracle_int_weight": (U64, [F32]),
                "oracle_row_weights": (I32, [P, I64, F32, P, P]),
                "oracle_philox4x32_10": (None, [P, P, P]),
                "oracle_uniforms": (None, [U64, U64, U32, U32, P]),
                "oracle_accept_decide": (I32, [U64, U64, U64, U64, U32]),
                "oracle_residual_pick": (I64, [P, U64, P, U64, I64, U32]),
                "oracle_weight_pick": (I64, [P, U64, I64, U32]),
                "oracle_accept_stochastic": (I32, [P, P, P, I32, I32, I64, F32,
                                                   U64, P, P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(P)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# fp16 helpers (the compiler's binary16 type)
# --------------------------------------------------------------------------
def f64_to_f16_bits(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f64_to_f16(_p(x), x.size, _p(out))
    return out


def f16_bits_to_f64(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float64)
    lib().oracle_f16_to_f64(_p(h), h.size, _p(out))
    return out


# --------------------------------------------------------------------------
# Model math
# --------------------------------------------------------------------------
class QWeight:
    """Canonical planes of one block-quantised matrix [N][K] (host numpy)."""

    def __init__(self, qtype: int, qs, qh, scales, N: int, K: int):
        assert qtype in (4, 6, 8) and K % 32 == 0
        self.qtype, self.N, self.K = qtype, int(N), int(K)
        self.qs = _c(qs, np.uint8).reshape(N, K // 32, 32 if qtype == 8 else 16)
        self.qh = None if qtype != 6 else _c(qh, np.uint8).reshape(N, K // 32, 8)
        self.scales = _c(scales, np.uint16).reshape(N, K // 32)

    def _struct(self) -> _QW:
        return _QW(self.qtype, _p(self.qs).value,
                   None if self.qh is None else _p(self.qh).value,
                   _p(self.scales).value, self.N, self.K)


def dequant(w: QWeight, n0: int = 0, rows: int | None = None) -> np.ndarray:
    rows = w.N - n0 if rows is None else rows
    out = np.empty((rows, w.K), np.float32)
    lib().oracle_dequant(w.qtype, _p(w.qs), None if w.qh is None else _p(w.qh),
                         _p(w.scales), w.N, w.K, n0, rows, _p(out))
    return out


def linear(w: QWeight, x_f16_bits) -> np.ndarray:
    """y[R][N] fp32 = fp64 sum over k of w[n][k] * x[r][k]; x is fp16 bits [R][K]."""
    x = _c(x_f16_bits, np.uint16)
    R = x.shape[0]
    assert x.shape[1] == w.K
    y = np.empty((R, w.N), np.float32)
    lib().oracle_linear(w.qtype, _p(w.qs), None if w.qh is None else _p(w.qh),
                        _p(w.scales), w.N, w.K, _p(x), R, _p(y))
    return y


def rmsnorm(h, gamma, eps: float) -> np.ndarray:
    h = _c(h, np.float32)
    gamma = _c(gamma, np.float32)
    out = np.empty(h.shape, np.uint16)
    lib().oracle_rmsnorm(_p(h), _p(gamma), h.shape[0], h.shape[1], eps, _p(out))
    return out


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotate-half RoPE of head vectors x[rows][hd] at positions pos[rows] -> fp16 bits."""
    x = _c(x, np.float32)
    pos = _c(pos, np.int64)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_rope(_p(x), x.shape[0], x.shape[1], _p(pos), theta, _p(out))
    return out


def attention(q_bits, kcache_bits, vcache_bits, pos) -> np.ndarray:
    """q[rows][nq][hd] fp16 bits; caches [nkv][max_ctx][hd] fp16 bits of one
    sequence; pos[rows] absolute positions.  Returns fp16 bits [rows][nq][hd]."""
    q = _c(q_bits, np.uint16)
    kc = _c(kcache_bits, np.uint16)
    vc = _c(vcache_bits, np.uint16)
    pos = _c(pos, np.int64)
    rows, nq, hd = q.shape
    nkv, max_ctx, _ = kc.shape
    out = np.empty(q.shape, np.uint16)
    lib().oracle_attention(_p(q), rows, nq, nkv, hd, _p(kc), _p(vc), max_ctx,
                           _p(pos), _p(out))
    return out


def swiglu(g, u) -> np.ndarray:
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    out = np.empty(g.shape, np.uint16)
    lib().oracle_swiglu(_p(g), _p(u), g.size, _p(out))
    return out


class Model:
    """Host copy of a synthetic decoder: canonical weights + descriptor."""

    def __init__(self, n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn,
                 vocab, max_ctx, embed_bits, norm_w, wqkv, wo, wgu, wd, lm_head,
                 rms_eps=1e-6, rope_theta=10000.0, use_rope=True):
        self.desc = _Desc(n_layers, hidden, n_q_heads, n_kv_heads, head_dim,
                          ffn, vocab, max_ctx, rms_eps, rope_theta, int(use_rope))
        self.embed = _c(embed_bits, np.uint16)
        self.norm_w = _c(norm_w, np.float32)
        self.wqkv, self.wo, self.wgu, self.wd = wqkv, wo, wgu, wd
        self.lm_head = lm_head

    def forward(self, tokens, n_past, kcache, vcache) -> np.ndarray:
        """tokens[n_seq][nt] int32; n_past[n_seq]; caches
        [L][n_seq][nkv][max_ctx][hd] fp16 bits, updated in place.
        Returns logits [n_seq*nt][V] fp32."""
        tokens = _c(tokens, np.int32)
        n_seq, nt = tokens.shape
        n_past = _c(n_past, np.int64)
        assert kcache.flags["C_CONTIGUOUS"] and vcache.flags["C_CONTIGUOUS"]
        assert kcache.dtype == np.uint16 and vcache.dtype == np.uint16
        L = self.desc.n_layers
        arr = lambda ws: (_QW * max(L, 1))(*[w._struct() for w in ws])
        a_qkv, a_o, a_gu, a_d = arr(self.wqkv), arr(self.wo), arr(self.wgu), arr(self.wd)
        lm = self.lm_head._struct()
        logits = np.empty((n_seq * nt, self.desc.vocab), np.float32)
        lib().oracle_forward(ctypes.byref(self.desc), _p(self.embed),
                             _p(self.norm_w), a_qkv, a_o, a_gu, a_d,
                             ctypes.byref(lm), n_seq, nt, _p(tokens), _p(n_past),
                             _p(kcache), _p(vcache), _p(logits))
        return logits


# --------------------------------------------------------------------------
# Accept
# --------------------------------------------------------------------------
def argmax(row) -> int:
    row = _c(row, np.float32)
    return int(lib().oracle_argmax(_p(row), row.size))


def accept_greedy(argmax_ids, draft):
    am = _c(argmax_ids, np.int32)
    dr = _c(draft, np.int32)
    n_seq, d1 = am.shape
    d = d1 - 1
    dr = dr.reshape(n_seq, d)
    n_acc = np.zeros(n_seq, np.int32)
    em = np.empty((n_seq, d + 1), np.int32)
    rc = lib().oracle_accept_greedy(_p(am), _p(dr), n_seq, d, _p(n_acc), _p(em))
    if rc != 0:
        raise ValueError("argmax row holds a NaN (negative id)")
    return n_acc, em


def exp_own(x: float) -> float:
    return float(lib().oracle_exp_own(float(x)))


def int_weight(x: float) -> int:
    return int(lib().oracle_int_weight(float(x)))


def row_weights(logits, T: float):
    lg = _c(logits, np.float32)
    W = np.empty(lg.size, np.uint64)
    S = ctypes.c_uint64(0)
    rc = lib().oracle_row_weights(_p(lg), lg.size, float(T), _p(W), ctypes.byref(S))
    if rc != 0:
        raise ValueError("non-finite logit")
    return W, int(S.value)


def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.empty(4, np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniforms(seed: int, slot: int, seq_id: int, domain: int):
    out = np.empty(4, np.uint32)
    lib().oracle_uniforms(seed, slot, seq_id, domain, _p(out))
    return out


def accept_decide(Wx: int, S: int, Wqx: int, Sq: int, U1: int) -> bool:
    return bool(lib().oracle_accept_decide(Wx, S, Wqx, Sq, U1))


def residual_pick(W, S: int, Wq, Sq: int, U2: int) -> int:
    W = _c(W, np.uint64)
    Wq = _c(Wq, np.uint64)
    return int(lib().oracle_residual_pick(_p(W), S, _p(Wq), Sq, W.size, U2))


def weight_pick(W, S: int, U2: int) -> int:
    W = _c(W, np.uint64)
    return int(lib().oracle_weight_pick(_p(W), S, W.size, U2))


def accept_stochastic(p_logits, q_logits, draft, T: float, seed: int, seq_ids,
                      emit_idx):
    """p_logits[n_seq][d+1][V], q_logits[n_seq][d][V], draft[n_seq][d].
    Returns (n_acc, emitted, new emit_idx)."""
    p = _c(p_logits, np.float32)
    n_seq, d1, V = p.shape
    d = d1 - 1
    q = _c(q_logits, np.float32).reshape(n_seq, d, V) if d > 0 else np.zeros((n_seq, 0, V), np.float32)
    dr = _c(draft, np.int32).reshape(n_seq, d)
    sid = _c(seq_ids, np.int32)
    ei = _c(emit_idx, np.uint64).copy()
    n_acc = np.zeros(n_seq, np.int32)
    em = np.empty((n_seq, d + 1), np.int32)
    rc = lib().oracle_accept_stochastic(_p(p), _p(q), _p(dr), n_seq, d, V,
                                        float(T), seed, _p(sid), _p(ei),
                                        _p(n_acc), _p(em))
    if rc != 0:
        raise ValueError("non-finite logit or draft id out of range")
    return n_acc, em, ei
