"""Python binding of the verify-round library (libspecverify.so, sm_103a).

Argument marshalling only: every step of the verify round runs in the CUDA
kernels behind the C ABI declared in ``include/spec_verify.h``.  torch is used
for device memory and streams.  There is no CPU fallback: if the compiled
library is missing, loading fails loudly.

Functions keep the C names (``spec_linear_q``, ``spec_verify_round``, ...);
tensors are passed as device pointers, streams as ``torch.cuda.Stream`` (or
None for torch's current stream).
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libspecverify.so")

SPEC_OK = 0
SPEC_E_INVALID = -1
SPEC_E_SHAPE = -2
SPEC_E_CUDA = -3
SPEC_E_OOM = -4
SPEC_E_UNSUPPORTED = -5
SPEC_E_TIMEOUT = -6
SPEC_Q4, SPEC_Q6, SPEC_Q8 = 4, 6, 8
SPEC_MAX_NT = 16
SPEC_PROF_QKV, SPEC_PROF_O, SPEC_PROF_GATE_UP, SPEC_PROF_DOWN = 0, 1, 2, 3
SPEC_PROF_LM_HEAD, SPEC_PROF_ALL_GEMMS, SPEC_PROF_ATTN = 4, 5, 6

EXPORTED = ["spec_last_error", "spec_qmat_create", "spec_qmat_destroy", "spec_linear_q",
            "spec_linear_q_tc", "spec_model_set_tc_min_seqs",
            "spec_model_create", "spec_model_destroy", "spec_model_kv_cache", "spec_kv_fill",
            "spec_kv_read", "spec_model_debug_read",
            "spec_state_set", "spec_state_get", "spec_error_check", "spec_model_set_graphs",
            "spec_model_set_wait_budget", "spec_model_profile", "spec_model_profile_read",
            "spec_verify_attn", "spec_lm_head", "spec_accept_greedy",
            "spec_accept_stochastic", "spec_accept_stochastic_noalloc", "spec_verify_round",
            "spec_verify_round_host", "spec_depth_params_default", "spec_depth_ctl_create",
            "spec_depth_ctl_destroy", "spec_depth_ctl_next", "spec_depth_ctl_observe",
            "spec_depth_ctl_estimates"]

P = ctypes.c_void_p
I32 = ctypes.c_int32
U64 = ctypes.c_uint64


class SpecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"spec error {code}: {msg}")
        self.code = code


class spec_qweight(ctypes.Structure):
    _fields_ = [("qtype", I32), ("N", I32), ("K", I32), ("qs", P), ("qh", P), ("scales", P)]


class spec_model_desc(ctypes.Structure):
    _fields_ = [("n_layers", I32), ("hidden", I32), ("n_q_heads", I32), ("n_kv_heads", I32),
                ("head_dim", I32), ("ffn", I32), ("vocab", I32), ("max_ctx", I32),
                ("max_nt", I32), ("max_seqs", I32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("use_rope", I32)]


class spec_model_weights(ctypes.Structure):
    _fields_ = [("embed", P), ("norm_w", P), ("wqkv", ctypes.POINTER(spec_qweight)),
                ("wo", ctypes.POINTER(spec_qweight)), ("wgu", ctypes.POINTER(spec_qweight)),
                ("wd", ctypes.POINTER(spec_qweight)), ("lm_head", spec_qweight)]


class spec_depth_params(ctypes.Structure):
    _fields_ = [("d_min", I32), ("d_max", I32), ("prior_accept", ctypes.c_double),
                ("prior_reject", ctypes.c_double), ("decay", ctypes.c_double),
                ("hysteresis", ctypes.c_double), ("cost_window", I32)]


class spec_sampling(ctypes.Structure):
    _fields_ = [("greedy", I32), ("temperature", ctypes.c_float), ("seed", U64)]


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            sig = {
                "spec_last_error": (None, [ctypes.c_char_p, ctypes.c_size_t]),
                "spec_qmat_create": (I32, [ctypes.POINTER(spec_qweight), I32, P, ctypes.POINTER(P)]),
                "spec_qmat_destroy": (I32, [P]),
                "spec_linear_q": (I32, [P, P, I32, P, P]),
                "spec_linear_q_tc": (I32, [P, P, I32, P, P]),
                "spec_model_set_tc_min_seqs": (I32, [P, I32]),
                "spec_model_create": (I32, [ctypes.POINTER(spec_model_desc),
                                            ctypes.POINTER(spec_model_weights), P, ctypes.POINTER(P)]),
                "spec_model_destroy": (I32, [P]),
                "spec_model_kv_cache": (I32, [P, I32, ctypes.POINTER(P), ctypes.POINTER(P)]),
                "spec_kv_fill": (I32, [P, I32, I32, I32, I32, P, P, P]),
                "spec_kv_read": (I32, [P, I32, I32, I32, I32, P, P, P]),
                "spec_model_debug_read": (I32, [P, I32, P, ctypes.c_size_t, P]),
                "spec_state_set": (I32, [P, I32, P, P, P, P]),
                "spec_state_get": (I32, [P, I32, P, P, P, P]),
                "spec_error_check": (I32, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
                "spec_model_set_graphs": (I32, [P, I32]),
                "spec_model_set_wait_budget": (I32, [P, I32]),
                "spec_model_profile": (I32, [P, I32]),
                "spec_model_profile_read": (I32, [P, I32, ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_int64),
                                                  ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_double)]),
                "spec_verify_attn": (I32, [P, I32, I32, P, I32, P, P, P, P, P]),
                "spec_lm_head": (I32, [P, P, I32, P, P, P]),
                "spec_accept_greedy": (I32, [P, P, I32, I32, P, P, P]),
                "spec_accept_stochastic": (I32, [P, P, P, I32, I32, I32, ctypes.c_float, U64,
                                                 P, P, P, P, P]),
                "spec_accept_stochastic_noalloc": (I32, [P, P, P, I32, I32, I32, ctypes.c_float,
                                                         U64, P, P, P, P, P]),
                "spec_verify_round": (I32, [P, I32, P, P, I32, P, ctypes.POINTER(spec_sampling),
                                            P, P, P, P]),
                "spec_verify_round_host": (I32, [P, I32, P, P, I32, P,
                                                 ctypes.POINTER(spec_sampling), P, P, P]),
                "spec_depth_params_default": (None, [ctypes.POINTER(spec_depth_params)]),
                "spec_depth_ctl_create": (I32, [ctypes.POINTER(spec_depth_params),
                                                ctypes.POINTER(P)]),
                "spec_depth_ctl_destroy": (I32, [P]),
                "spec_depth_ctl_next": (I32, [P, ctypes.POINTER(I32)]),
                "spec_depth_ctl_observe": (I32, [P, I32, I32, P, ctypes.c_double,
                                                 ctypes.POINTER(I32)]),
                "spec_depth_ctl_estimates": (I32, [P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def last_error() -> str:
    buf = ctypes.create_string_buffer(1024)
    lib().spec_last_error(buf, 1024)
    return buf.value.decode(errors="replace")


def _check(rc: int):
    if rc != SPEC_OK:
        raise SpecError(rc, last_error())


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _qweight(w: dict) -> spec_qweight:
    """dict(qtype, N, K, qs, qh, scales) of device tensors -> spec_qweight."""
    return spec_qweight(int(w["qtype"]), int(w["N"]), int(w["K"]), w["qs"].data_ptr(),
                        None if w.get("qh") is None else w["qh"].data_ptr(),
                        w["scales"].data_ptr())


# ---------------------------------------------------------------------------
# packed matrices and the verify GEMM
# ---------------------------------------------------------------------------
class QMat:
    """A block-quantised matrix repacked on the device (spec_qmat)."""

    def __init__(self, w: dict, max_rows: int = SPEC_MAX_NT, stream=None):
        self.handle = P()
        self.N, self.K, self.qtype = int(w["N"]), int(w["K"]), int(w["qtype"])
        qw = _qweight(w)
        _check(lib().spec_qmat_create(ctypes.byref(qw), int(max_rows), _stream(stream),
                                      ctypes.byref(self.handle)))

    def close(self):
        if self.handle:
            lib().spec_qmat_destroy(self.handle)
            self.handle = P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spec_qmat_create(w: dict, max_rows: int = SPEC_MAX_NT, stream=None) -> QMat:
    return QMat(w, max_rows, stream)


def spec_linear_q(w: QMat, x, nt: int, y, stream=None):
    """y[nt][N] fp32 = W x[nt][K] (fp16); all device tensors."""
    _check(lib().spec_linear_q(w.handle, _ptr(x), int(nt), _ptr(y), _stream(stream)))


def spec_linear_q_tc(w: QMat, x, R: int, y, stream=None):
    """The same product on the tensor-core GEMM of multi-sequence rounds."""
    _check(lib().spec_linear_q_tc(w.handle, _ptr(x), int(R), _ptr(y), _stream(stream)))


# ---------------------------------------------------------------------------
# the decoder model
# ---------------------------------------------------------------------------
class Model:
    """spec_model: repacked weights, KV cache, per-sequence state."""

    def __init__(self, desc: dict, weights: dict, stream=None):
        d = spec_model_desc(int(desc["n_layers"]), int(desc["hidden"]),
                            int(desc.get("n_q_heads", 1)), int(desc.get("n_kv_heads", 1)),
                            int(desc.get("head_dim", 128)), int(desc.get("ffn", 32)),
                            int(desc["vocab"]), int(desc.get("max_ctx", 1)),
                            int(desc.get("max_nt", SPEC_MAX_NT)), int(desc.get("max_seqs", 1)),
                            float(desc.get("rms_eps", 1e-6)),
                            float(desc.get("rope_theta", 10000.0)),
                            int(desc.get("use_rope", 1)))
        self.desc = d
        L = d.n_layers
        arr = lambda key: (spec_qweight * max(L, 1))(*[_qweight(w) for w in weights.get(key, [])])
        self._keep = [arr("wqkv"), arr("wo"), arr("wgu"), arr("wd")]
        W = spec_model_weights(
            None if weights.get("embed") is None else weights["embed"].data_ptr(),
            weights["norm_w"].data_ptr(), self._keep[0], self._keep[1], self._keep[2],
            self._keep[3], _qweight(weights["lm_head"]))
        self.handle = P()
        _check(lib().spec_model_create(ctypes.byref(d), ctypes.byref(W), _stream(stream),
                                       ctypes.byref(self.handle)))

    def close(self):
        if self.handle:
            lib().spec_model_destroy(self.handle)
            self.handle = P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_cache(self, layer: int):
        """(k, v) device pointers (ints) of one layer's cache
        [max_seqs][n_kv_heads][max_ctx][head_dim] fp16."""
        k, v = P(), P()
        _check(lib().spec_model_kv_cache(self.handle, int(layer), ctypes.byref(k), ctypes.byref(v)))
        return k.value, v.value

    def set_graphs(self, enable: bool):
        _check(lib().spec_model_set_graphs(self.handle, int(bool(enable))))

    def set_tc_min_seqs(self, min_seqs: int):
        """Rounds of at least min_seqs sequences use the tensor-core GEMM (0: never)."""
        _check(lib().spec_model_set_tc_min_seqs(self.handle, int(min_seqs)))

    def profile(self, enable: bool):
        """In-round kernel timing on (raw launches, events around each GEMM and
        attention launch) or off; clears the totals."""
        _check(lib().spec_model_profile(self.handle, int(bool(enable))))

    def profile_read(self, kind: int) -> dict:
        """Totals of one kernel class since the last profile() call."""
        t, b, f = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        n = ctypes.c_int64()
        _check(lib().spec_model_profile_read(self.handle, int(kind), ctypes.byref(t),
                                             ctypes.byref(n), ctypes.byref(b), ctypes.byref(f)))
        return dict(seconds=t.value, launches=n.value, bytes=b.value, flops=f.value)

    def set_wait_budget(self, tries: int):
        """Test hook: try budget of each GEMM CTA's first copy wait (see the header)."""
        _check(lib().spec_model_set_wait_budget(self.handle, int(tries)))


def spec_kv_fill(m: Model, layer: int, seq: int, pos0: int, n_pos: int, k, v, stream=None):
    """k, v: fp16 tensors [n_kv_heads][n_pos][head_dim] (device or pinned host)."""
    _check(lib().spec_kv_fill(m.handle, int(layer), int(seq), int(pos0), int(n_pos), _ptr(k),
                              _ptr(v), _stream(stream)))


def spec_kv_read(m: Model, layer: int, seq: int, pos0: int, n_pos: int, k, v, stream=None):
    """Copies cache rows out into k, v: fp16 tensors [n_kv_heads][n_pos][head_dim]."""
    _check(lib().spec_kv_read(m.handle, int(layer), int(seq), int(pos0), int(n_pos), _ptr(k),
                              _ptr(v), _stream(stream)))


def spec_model_debug_read(m: Model, which: int, dst, stream=None):
    """Copies an internal activation buffer of the last pass into dst."""
    _check(lib().spec_model_debug_read(m.handle, int(which), _ptr(dst),
                                       dst.numel() * dst.element_size(), _stream(stream)))


def _host_array(values, ctype):
    if values is None:
        return None
    vals = [int(v) for v in values]
    return (ctype * len(vals))(*vals)


def spec_state_set(m: Model, seq_ids, n_past=None, emit_idx=None, anchor=None):
    n = len(seq_ids)
    _check(lib().spec_state_set(m.handle, n, _host_array(seq_ids, ctypes.c_int32),
                                _host_array(n_past, ctypes.c_int32),
                                _host_array(emit_idx, ctypes.c_uint64),
                                _host_array(anchor, ctypes.c_int32)))


def spec_state_get(m: Model, seq_ids):
    n = len(seq_ids)
    a = (ctypes.c_int32 * n)()
    b = (ctypes.c_uint64 * n)()
    c = (ctypes.c_int32 * n)()
    _check(lib().spec_state_get(m.handle, n, _host_array(seq_ids, ctypes.c_int32), a, b, c))
    return list(a), list(b), list(c)


def spec_error_check(m: Model | None = None, stream=None) -> int:
    """Synchronises, returns and clears the device error bits (0 = none)."""
    bits = ctypes.c_uint32(0)
    rc = lib().spec_error_check(None if m is None else m.handle, _stream(stream),
                                ctypes.byref(bits))
    if rc not in (SPEC_OK, SPEC_E_INVALID):
        _check(rc)
    return int(bits.value)


def spec_verify_attn(m: Model, layer: int, n_seq: int, seq_ids, nt: int, q, k_new, v_new, out,
                     stream=None):
    _check(lib().spec_verify_attn(m.handle, int(layer), int(n_seq), _ptr(seq_ids), int(nt),
                                  _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _stream(stream)))


def spec_lm_head(m: Model, x, R: int, logits=None, argmax=None, stream=None):
    _check(lib().spec_lm_head(m.handle, _ptr(x), int(R), _ptr(logits), _ptr(argmax),
                              _stream(stream)))


def spec_accept_greedy(argmax, draft, n_seq: int, d: int, n_acc, emitted, stream=None):
    _check(lib().spec_accept_greedy(_ptr(argmax), _ptr(draft), int(n_seq), int(d), _ptr(n_acc),
                                    _ptr(emitted), _stream(stream)))


def spec_accept_stochastic(p_logits, q_logits, draft, n_seq: int, d: int, V: int,
                           temperature: float, seed: int, seq_ids, emit_idx, n_acc, emitted,
                           stream=None):
    _check(lib().spec_accept_stochastic(_ptr(p_logits), _ptr(q_logits), _ptr(draft), int(n_seq),
                                        int(d), int(V), float(temperature), int(seed),
                                        _ptr(seq_ids), _ptr(emit_idx), _ptr(n_acc),
                                        _ptr(emitted), _stream(stream)))


def spec_accept_stochastic_noalloc(p_logits, q_logits, draft, n_seq: int, d: int, V: int,
                                   temperature: float, seed: int, seq_ids, emit_idx, n_acc,
                                   emitted, stream=None):
    """spec_accept_stochastic without any allocation (fixed scratch; see the header)."""
    _check(lib().spec_accept_stochastic_noalloc(_ptr(p_logits), _ptr(q_logits), _ptr(draft),
                                                int(n_seq), int(d), int(V), float(temperature),
                                                int(seed), _ptr(seq_ids), _ptr(emit_idx),
                                                _ptr(n_acc), _ptr(emitted), _stream(stream)))


def spec_verify_round(m: Model, n_seq: int, seq_ids, draft, d: int, q_logits=None,
                      greedy: bool = True, temperature: float = 1.0, seed: int = 0,
                      n_acc=None, emitted=None, logits_out=None, stream=None):
    sp = spec_sampling(int(bool(greedy)), float(temperature), int(seed))
    _check(lib().spec_verify_round(m.handle, int(n_seq), _ptr(seq_ids), _ptr(draft), int(d),
                                   _ptr(q_logits), ctypes.byref(sp), _ptr(n_acc), _ptr(emitted),
                                   _ptr(logits_out), _stream(stream)))


def _host_i32(a, n, name):
    """a as a C-contiguous int32 numpy array of at least n elements (no copy
    when it already is one)."""
    import numpy as np
    if not (type(a) is np.ndarray and a.dtype == np.int32 and a.flags.c_contiguous):
        a = np.ascontiguousarray(a, dtype=np.int32)
    if a.size < n:
        raise ValueError(f"{name}: {n} int32 values required, got {a.size}")
    return a


def spec_verify_round_host(m: Model, n_seq: int, seq_ids, draft, d: int, q_logits=None,
                           greedy: bool = True, temperature: float = 1.0, seed: int = 0,
                           n_acc=None, emitted=None, stream=None):
    """spec_verify_round with host (numpy int32) seq_ids, draft, n_acc and emitted;
    q_logits a device tensor, a (pinned) host tensor or a float32 numpy array.
    Returns (n_acc, emitted); they are valid on return (the call synchronises).
    n_acc / emitted, when given, must be C-contiguous int32 arrays (written in
    place)."""
    import numpy as np
    sid = _host_i32(seq_ids, n_seq, "seq_ids")
    dr = _host_i32(draft, n_seq * d, "draft") if d > 0 else None
    if n_acc is None:
        n_acc = np.empty(n_seq, np.int32)
    if emitted is None:
        emitted = np.empty((n_seq, d + 1), np.int32)
    for a, n, name in ((n_acc, n_seq, "n_acc"), (emitted, n_seq * (d + 1), "emitted")):
        if not (type(a) is np.ndarray and a.dtype == np.int32 and a.flags.c_contiguous
                and a.size >= n):
            raise ValueError(f"{name}: a C-contiguous int32 numpy array of {n} values is required")
    sp = spec_sampling(int(bool(greedy)), float(temperature), int(seed))
    if type(q_logits) is np.ndarray:  # host q_logits: copied by the library
        if not (q_logits.dtype == np.float32 and q_logits.flags.c_contiguous):
            raise ValueError("q_logits: a C-contiguous float32 array is required")
        qp = ctypes.c_void_p(q_logits.ctypes.data)
    else:
        qp = _ptr(q_logits)
    _check(lib().spec_verify_round_host(m.handle, int(n_seq), sid.ctypes.data,
                                        None if dr is None else dr.ctypes.data, int(d),
                                        qp, ctypes.byref(sp), n_acc.ctypes.data,
                                        emitted.ctypes.data, _stream(stream)))
    return n_acc, emitted


class DepthController:
    """The library's adaptive draft-depth controller (host only; rules in
    include/spec_verify.h).  Keyword arguments override the defaults."""

    def __init__(self, **kw):
        prm = spec_depth_params()
        lib().spec_depth_params_default(ctypes.byref(prm))
        for k, v in kw.items():
            setattr(prm, k, v)
        self.params = prm
        h = P()
        _check(lib().spec_depth_ctl_create(ctypes.byref(prm), ctypes.byref(h)))
        self.handle = h

    def next_depth(self) -> int:
        d = I32()
        _check(lib().spec_depth_ctl_next(self.handle, ctypes.byref(d)))
        return d.value

    def observe(self, d: int, n_acc, round_seconds: float) -> int:
        import numpy as np
        a = np.ascontiguousarray(n_acc, dtype=np.int32)
        nd = I32()
        _check(lib().spec_depth_ctl_observe(self.handle, int(d), int(a.size),
                                            a.ctypes.data if a.size else None,
                                            float(round_seconds), ctypes.byref(nd)))
        return nd.value

    def estimates(self):
        """(p[0..d_max], r[0..d_max]) as lists of floats."""
        n = self.params.d_max + 1
        p = (ctypes.c_double * n)()
        r = (ctypes.c_double * n)()
        _check(lib().spec_depth_ctl_estimates(self.handle, p, r))
        return list(p), list(r)

    def close(self):
        if self.handle:
            lib().spec_depth_ctl_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
