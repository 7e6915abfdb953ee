"""Plain float64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The
product path never touches it, and it shares no code with the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C, float64, sequential loops in
index order, its own Philox4x32-10). This module only compiles it with gcc and
marshals numpy arrays through ctypes. Every function documents the page passage
it follows; see the header of ``oracle.c`` for the sources and readings.

Parity status of each function (what pins it; see tests/test_oracle_pins.py):
  philox4x32_10 / uniform_pair   -- pinned: the generator's published
                                    known-answer vectors (zero, all-ones,
                                    pi digits) and Triton's independent
                                    Philox (CPU interpreter)
  softmax_row / normalize_row    -- pinned: scipy.special.softmax, closed forms
  residual                       -- pinned: the page's worked example, the
                                    identity Z = 1 - sum min(p, q)
  inverse_cdf                    -- pinned: brute force over the u-grid
  argmax_row                     -- pinned: numpy argmax (NaN -> -inf)
  verify_sample                  -- pinned: exact enumeration, chi-square,
                                    expected-tokens formula, page's statistical test
  verify_greedy / kv_rollback    -- pinned: brute force, special cases
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
SEQ_OK, SEQ_BAD_TOKEN, SEQ_BAD_KV, SEQ_BAD_ROW, SEQ_BAD_LAYOUT, SEQ_BAD_TEMP = 0, 1, 2, 3, 4, 5
SEQ_UNSUPPORTED = 7


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fast-math: IEEE float64)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-D_GNU_SOURCE", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OrcArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("gamma_max", ctypes.c_int32),
        ("rows_target", ctypes.c_int64), ("rows_draft", ctypes.c_int64),
        ("target_row_off", ctypes.c_void_p), ("draft_row_off", ctypes.c_void_p),
        ("target", ctypes.c_void_p), ("target_dtype", ctypes.c_int32),
        ("draft", ctypes.c_void_p), ("draft_dtype", ctypes.c_int32),
        ("draft_is_probs", ctypes.c_int32),
        ("draft_tokens", ctypes.c_void_p),
        ("temperatures", ctypes.c_void_p), ("temperature", ctypes.c_float),
        ("seed", ctypes.c_uint64), ("round", ctypes.c_uint64), ("seq_offset", ctypes.c_uint32),
        ("uniforms", ctypes.c_void_p),
        ("kv_in", ctypes.c_void_p), ("block_size", ctypes.c_int32),
        ("out_tokens", ctypes.c_void_p), ("out_accepted", ctypes.c_void_p),
        ("kv_out", ctypes.c_void_p), ("out_blocks", ctypes.c_void_p), ("seq_status", ctypes.c_void_p),
        ("diag_acc_margin", ctypes.c_void_p), ("diag_u_smp", ctypes.c_void_p),
        ("diag_cdf_lo", ctypes.c_void_p), ("diag_cdf_hi", ctypes.c_void_p), ("diag_z", ctypes.c_void_p),
        ("top_k", ctypes.c_int32), ("top_ks", ctypes.c_void_p),
        ("top_p", ctypes.c_float), ("top_ps", ctypes.c_void_p),
    ]


class OrcTreeArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("greedy", ctypes.c_int32),
        ("nodes", ctypes.c_int64),
        ("node_off", ctypes.c_void_p), ("parent", ctypes.c_void_p), ("tokens", ctypes.c_void_p),
        ("target", ctypes.c_void_p), ("target_dtype", ctypes.c_int32),
        ("draft", ctypes.c_void_p), ("draft_dtype", ctypes.c_int32), ("draft_is_probs", ctypes.c_int32),
        ("temperatures", ctypes.c_void_p), ("temperature", ctypes.c_float),
        ("seed", ctypes.c_uint64), ("round", ctypes.c_uint64), ("seq_offset", ctypes.c_uint32),
        ("out_tokens", ctypes.c_void_p), ("out_accepted", ctypes.c_void_p), ("out_path", ctypes.c_void_p),
        ("seq_status", ctypes.c_void_p),
        ("diag_acc_margin", ctypes.c_void_p), ("diag_u_smp", ctypes.c_void_p),
        ("diag_cdf_lo", ctypes.c_void_p), ("diag_cdf_hi", ctypes.c_void_p),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            vp, i32, i64, u32, u64, dbl = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                         ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double)
            L.orc_value.restype = dbl
            L.orc_value.argtypes = [vp, i32, i64]
            L.orc_philox4x32_10.restype = None
            L.orc_philox4x32_10.argtypes = [vp, vp, vp]
            L.orc_uniform_pair.restype = None
            L.orc_uniform_pair.argtypes = [u64, u64, u32, u32, vp, vp]
            L.orc_softmax_row.restype = i32
            L.orc_softmax_row.argtypes = [vp, i32, i64, dbl, vp]
            L.orc_normalize_row.restype = i32
            L.orc_normalize_row.argtypes = [vp, i32, i64, vp]
            L.orc_topk_threshold.restype = dbl
            L.orc_topk_threshold.argtypes = [vp, i32, i64, i64]
            L.orc_topp_threshold.restype = dbl
            L.orc_topp_threshold.argtypes = [vp, i32, i64, dbl, i32, dbl, dbl]
            L.orc_softmax_row_topk.restype = i32
            L.orc_softmax_row_topk.argtypes = [vp, i32, i64, dbl, dbl, vp]
            L.orc_normalize_row_topk.restype = i32
            L.orc_normalize_row_topk.argtypes = [vp, i32, i64, dbl, vp]
            L.orc_acceptance_ema.restype = None
            L.orc_acceptance_ema.argtypes = [vp, vp, i32, i64, vp, ctypes.c_float, vp, vp]
            L.orc_speedups.restype = None
            L.orc_speedups.argtypes = [ctypes.c_float, i32, ctypes.c_float, vp]
            L.orc_best_gamma.restype = i32
            L.orc_best_gamma.argtypes = [ctypes.c_float, i32, ctypes.c_float]
            L.orc_adapt_gamma.restype = i64
            L.orc_adapt_gamma.argtypes = [vp, i64, i32, ctypes.c_float, i64, vp]
            L.orc_ngram_draft.restype = None
            L.orc_ngram_draft.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, vp, vp]
            L.orc_tree_verify.restype = None
            L.orc_tree_verify.argtypes = [ctypes.POINTER(OrcTreeArgs)]
            L.orc_residual.restype = dbl
            L.orc_residual.argtypes = [vp, vp, i64, vp]
            L.orc_inverse_cdf.restype = i64
            L.orc_inverse_cdf.argtypes = [vp, i64, dbl]
            L.orc_cdf_edges.restype = None
            L.orc_cdf_edges.argtypes = [vp, i64, i64, vp, vp]
            L.orc_argmax_row.restype = i64
            L.orc_argmax_row.argtypes = [vp, i32, i64]
            L.orc_verify_sample.restype = ctypes.c_int
            L.orc_verify_sample.argtypes = [ctypes.POINTER(OrcArgs), i32]
            L.orc_verify_greedy.restype = ctypes.c_int
            L.orc_verify_greedy.argtypes = [ctypes.POINTER(OrcArgs), i32]
            L.orc_kv_rollback.restype = None
            L.orc_kv_rollback.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp]
            L.orc_accept_terms.restype = i32
            L.orc_accept_terms.argtypes = [ctypes.POINTER(OrcArgs), i64, i64, vp, vp]
            L.orc_position_rows.restype = i32
            L.orc_position_rows.argtypes = [ctypes.POINTER(OrcArgs), i64, i64, vp, vp, vp, vp]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle rows must be float32 or uint16 (bf16 bits), got {a.dtype}")


# --------------------------------------------------------------------------- RNG
def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 block (SC'11 definition): 4 counter words, 2 key words -> 4 words."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def uniform_pair(seed: int, rnd: int, seq: int, pos: int):
    """(u_acc, u_smp) for one draw position: Philox key = seed, counter = (pos, seq, round)."""
    ua, us = ctypes.c_double(), ctypes.c_double()
    lib().orc_uniform_pair(seed, rnd, seq, pos, ctypes.byref(ua), ctypes.byref(us))
    return ua.value, us.value


# ----------------------------------------------------------------- distributions
def softmax_row(row: np.ndarray, T: float = 1.0):
    """softmax(l / T) of one logits row in float64. Returns (status, p)."""
    row = np.ascontiguousarray(row)
    p = np.zeros(row.shape[0], dtype=np.float64)
    st = lib().orc_softmax_row(row.ctypes.data, _dtype_code(row), row.shape[0], float(T), p.ctypes.data)
    return st, p


def normalize_row(row: np.ndarray):
    """A probability row divided by its own sum. Returns (status, q)."""
    row = np.ascontiguousarray(row)
    q = np.zeros(row.shape[0], dtype=np.float64)
    st = lib().orc_normalize_row(row.ctypes.data, _dtype_code(row), row.shape[0], q.ctypes.data)
    return st, q


def topk_threshold(row: np.ndarray, k: int) -> float:
    """The k-th largest value of a row (NaN read as -inf); -inf when k <= 0 or k >= V."""
    row = np.ascontiguousarray(row)
    return float(lib().orc_topk_threshold(row.ctypes.data, _dtype_code(row), row.shape[0], int(k)))


def topp_threshold(row: np.ndarray, T: float, tau_k: float, top_p: float, probs: bool = False) -> float:
    """The top-p threshold over the columns >= tau_k (tau_k itself unless 0 < top_p < 1)."""
    row = np.ascontiguousarray(row)
    return float(lib().orc_topp_threshold(row.ctypes.data, _dtype_code(row), row.shape[0], float(T), int(probs),
                                          float(tau_k), float(top_p)))


def softmax_row_topk(row: np.ndarray, T: float, tau: float):
    """softmax(l / T) over the columns with l >= tau, 0 elsewhere. Returns (status, p)."""
    row = np.ascontiguousarray(row)
    p = np.zeros(row.shape[0], dtype=np.float64)
    st = lib().orc_softmax_row_topk(row.ctypes.data, _dtype_code(row), row.shape[0], float(T), float(tau),
                                    p.ctypes.data)
    return st, p


def normalize_row_topk(row: np.ndarray, tau: float):
    """A probability row kept where value >= tau, divided by the kept sum. Returns (status, q)."""
    row = np.ascontiguousarray(row)
    q = np.zeros(row.shape[0], dtype=np.float64)
    st = lib().orc_normalize_row_topk(row.ctypes.data, _dtype_code(row), row.shape[0], float(tau), q.ctypes.data)
    return st, q


def acceptance_ema(accepted, gammas, gamma_max, ema, lam, status=None):
    """One round's update of the running acceptance (float32 state)."""
    acc = np.ascontiguousarray(accepted, dtype=np.int32)
    g = None if gammas is None else np.ascontiguousarray(gammas, dtype=np.int32)
    st = None if status is None else np.ascontiguousarray(status, dtype=np.int32)
    e_in = np.ascontiguousarray(ema, dtype=np.float32)
    e_out = np.empty_like(e_in)
    lib().orc_acceptance_ema(acc.ctypes.data, _ptr(g), int(gamma_max), acc.shape[0], _ptr(st), float(lam),
                             e_in.ctypes.data, e_out.ctypes.data)
    return e_out


def speedups(alpha: float, gamma_max: int, c: float) -> np.ndarray:
    """E(alpha, g) / (1 + g c) for g = 0..gamma_max (float32 arithmetic)."""
    sp = np.zeros(int(gamma_max) + 1, dtype=np.float32)
    lib().orc_speedups(float(alpha), int(gamma_max), float(c), sp.ctypes.data)
    return sp


def best_gamma(ema: float, gamma_max: int, c: float) -> int:
    return int(lib().orc_best_gamma(float(ema), int(gamma_max), float(c)))


def adapt_gamma(ema, gamma_max: int, c: float, max_positions: int = 0):
    """(gammas int32 [B], verify positions of the chosen gammas before the switch)."""
    e = np.ascontiguousarray(ema, dtype=np.float32)
    out = np.zeros(e.shape[0], dtype=np.int32)
    tot = lib().orc_adapt_gamma(e.ctypes.data, e.shape[0], int(gamma_max), float(c), int(max_positions),
                                out.ctypes.data)
    return out, int(tot)


def ngram_draft(ctx, ctx_off, n_max: int, n_min: int, gamma: int):
    """Prompt-lookup drafts: dict of draft [B, gamma] (-1 padded), n_draft, match_pos, match_n."""
    c = np.ascontiguousarray(ctx, dtype=np.int32)
    off = np.ascontiguousarray(ctx_off, dtype=np.int64)
    B = off.shape[0] - 1
    draft = np.full(B * max(gamma, 1), -7, dtype=np.int32)
    nd = np.zeros(B, np.int32)
    pos = np.zeros(B, np.int64)
    mn = np.zeros(B, np.int32)
    lib().orc_ngram_draft(c.ctypes.data, off.ctypes.data, B, int(n_max), int(n_min), int(gamma), draft.ctypes.data,
                          nd.ctypes.data, pos.ctypes.data, mn.ctypes.data)
    return {"draft": draft[:B * gamma].reshape(B, gamma), "n_draft": nd, "match_pos": pos, "match_n": mn}


def tree_verify(w, *, seed=0, rnd=0, seq_offset=0, greedy=None, parent=None, tokens=None, diagnostics=False):
    """Tree verification of a workloads.TreeWorkload (float64; one thread)."""
    N, B = w.nodes, w.batch
    keep = []

    def arr(a, dt):
        a = np.ascontiguousarray(a, dtype=dt)
        keep.append(a)
        return a

    off = arr(w.node_off, np.int64)
    par = arr(w.parent if parent is None else parent, np.int32)
    tok = arr(w.tokens if tokens is None else tokens, np.int32)
    tgt = np.ascontiguousarray(w.target)
    dft = np.ascontiguousarray(w.draft)
    temps = None if w.temperatures is None else arr(w.temperatures, np.float32)
    out = {"tokens": np.full(N, -7, np.int32), "accepted": np.full(B, -7, np.int32),
           "path": np.full(N, -7, np.int32), "status": np.full(B, -7, np.int32)}
    diag = {k: np.full(B, np.nan) for k in ("acc_margin", "u_smp", "cdf_lo", "cdf_hi")} if diagnostics else None
    a = OrcTreeArgs()
    a.batch, a.vocab, a.nodes = B, w.vocab, min(par.shape[0], tok.shape[0], tgt.shape[0], dft.shape[0])
    a.greedy = int(w.greedy if greedy is None else greedy)
    a.node_off, a.parent, a.tokens = off.ctypes.data, par.ctypes.data, tok.ctypes.data
    a.target, a.target_dtype = tgt.ctypes.data, _dtype_code(tgt)
    a.draft, a.draft_dtype = dft.ctypes.data, _dtype_code(dft)
    a.draft_is_probs = int(w.draft_is_probs)
    a.temperatures = _ptr(temps)
    a.temperature = float(w.temperature)
    a.seed, a.round, a.seq_offset = int(seed) & (2**64 - 1), int(rnd) & (2**64 - 1), int(seq_offset)
    a.out_tokens, a.out_accepted = out["tokens"].ctypes.data, out["accepted"].ctypes.data
    a.out_path, a.seq_status = out["path"].ctypes.data, out["status"].ctypes.data
    if diag is not None:
        a.diag_acc_margin, a.diag_u_smp = diag["acc_margin"].ctypes.data, diag["u_smp"].ctypes.data
        a.diag_cdf_lo, a.diag_cdf_hi = diag["cdf_lo"].ctypes.data, diag["cdf_hi"].ctypes.data
        out["diag"] = diag
    lib().orc_tree_verify(ctypes.byref(a))
    return out


def residual(p: np.ndarray, q: np.ndarray):
    """r = max(0, p - q) and its sum Z."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    r = np.zeros_like(p)
    Z = lib().orc_residual(p.ctypes.data, q.ctypes.data, p.shape[0], r.ctypes.data)
    return r, Z


def inverse_cdf(w: np.ndarray, u: float) -> int:
    w = np.ascontiguousarray(w, dtype=np.float64)
    return int(lib().orc_inverse_cdf(w.ctypes.data, w.shape[0], float(u)))


def cdf_edges(w: np.ndarray, j: int):
    w = np.ascontiguousarray(w, dtype=np.float64)
    lo, hi = ctypes.c_double(), ctypes.c_double()
    lib().orc_cdf_edges(w.ctypes.data, w.shape[0], int(j), ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def argmax_row(row: np.ndarray) -> int:
    row = np.ascontiguousarray(row)
    return int(lib().orc_argmax_row(row.ctypes.data, _dtype_code(row), row.shape[0]))


def value(row: np.ndarray, j: int) -> float:
    row = np.ascontiguousarray(row)
    return float(lib().orc_value(row.ctypes.data, _dtype_code(row), int(j)))


# ------------------------------------------------------------------ batch verify
class _Call:
    """Holds the numpy buffers of one oracle call alive next to its OrcArgs."""

    def __init__(self, w, *, seed=0, rnd=0, seq_offset=0, uniforms=None, draft_tokens=None,
                 diagnostics=False):
        B = w.batch
        self.keep = []

        def keep(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            self.keep.append(a)
            return a

        tgt = keep(w.target)
        dft = keep(w.draft) if w.draft is not None else None
        toks = keep(np.asarray(draft_tokens if draft_tokens is not None else w.draft_tokens, dtype=np.int32))
        tro = keep(None if w.target_row_off is None else np.asarray(w.target_row_off, dtype=np.int64))
        dro = keep(None if w.draft_row_off is None else np.asarray(w.draft_row_off, dtype=np.int64))
        temps = keep(None if w.temperatures is None else np.asarray(w.temperatures, dtype=np.float32))
        kv = keep(None if w.kv_in is None else np.asarray(w.kv_in, dtype=np.int32))
        unif = keep(None if uniforms is None else np.asarray(uniforms, dtype=np.float32))
        topks = keep(None if getattr(w, "top_ks", None) is None else np.asarray(w.top_ks, dtype=np.int32))
        topps = keep(None if getattr(w, "top_ps", None) is None else np.asarray(w.top_ps, dtype=np.float32))
        self.out_tokens = np.full(w.rows_target, -7, dtype=np.int32)
        self.out_accepted = np.full(B, -7, dtype=np.int32)
        self.kv_out = np.full(B, -7, dtype=np.int32)
        self.out_blocks = np.full(B, -7, dtype=np.int32)
        self.seq_status = np.full(B, -7, dtype=np.int32)
        self.diag = None
        if diagnostics:
            self.diag = {k: np.full(B, np.nan) for k in ("acc_margin", "u_smp", "cdf_lo", "cdf_hi", "z")}
        a = OrcArgs()
        a.batch, a.vocab, a.gamma_max = B, w.vocab, w.gamma_max
        a.rows_target, a.rows_draft = w.rows_target, w.rows_draft
        a.target_row_off, a.draft_row_off = _ptr(tro), _ptr(dro)
        a.target, a.target_dtype = _ptr(tgt), _dtype_code(tgt)
        a.draft = _ptr(dft)
        a.draft_dtype = _dtype_code(dft) if dft is not None else F32
        a.draft_is_probs = int(w.draft_is_probs)
        a.draft_tokens = _ptr(toks)
        a.temperatures = _ptr(temps)
        a.temperature = float(w.temperature)
        a.seed, a.round, a.seq_offset = int(seed), int(rnd), int(seq_offset)
        a.uniforms = _ptr(unif)
        a.kv_in, a.block_size = _ptr(kv), int(w.block_size)
        a.out_tokens, a.out_accepted = _ptr(self.out_tokens), _ptr(self.out_accepted)
        a.kv_out = _ptr(self.kv_out) if kv is not None else None
        a.out_blocks = _ptr(self.out_blocks) if (kv is not None and w.block_size > 0) else None
        a.seq_status = _ptr(self.seq_status)
        a.top_k = int(getattr(w, "top_k", 0))
        a.top_ks = _ptr(topks)
        a.top_p = float(getattr(w, "top_p", 0.0))
        a.top_ps = _ptr(topps)
        if self.diag is not None:
            a.diag_acc_margin = _ptr(self.diag["acc_margin"])
            a.diag_u_smp = _ptr(self.diag["u_smp"])
            a.diag_cdf_lo = _ptr(self.diag["cdf_lo"])
            a.diag_cdf_hi = _ptr(self.diag["cdf_hi"])
            a.diag_z = _ptr(self.diag["z"])
        self.args = a
        self.has_kv = kv is not None
        self.has_blocks = kv is not None and w.block_size > 0

    def result(self):
        out = {"tokens": self.out_tokens, "accepted": self.out_accepted, "status": self.seq_status}
        if self.has_kv:
            out["kv"] = self.kv_out
        if self.has_blocks:
            out["blocks"] = self.out_blocks
        if self.diag is not None:
            out["diag"] = self.diag
        return out


def verify_sample(w, *, seed=0, rnd=0, seq_offset=0, uniforms=None, draft_tokens=None,
                  nthreads=1, diagnostics=False):
    """Sampling verify of a whole batch (``w`` is a workloads.Workload)."""
    c = _Call(w, seed=seed, rnd=rnd, seq_offset=seq_offset, uniforms=uniforms,
              draft_tokens=draft_tokens, diagnostics=diagnostics)
    lib().orc_verify_sample(ctypes.byref(c.args), int(nthreads))
    return c.result()


def verify_greedy(w, *, draft_tokens=None, nthreads=1):
    """Greedy verify of a whole batch."""
    c = _Call(w, draft_tokens=draft_tokens)
    lib().orc_verify_greedy(ctypes.byref(c.args), int(nthreads))
    return c.result()


def kv_rollback(kv_in, accepted, gammas, gamma_max, block_size=0):
    kv_in = np.ascontiguousarray(kv_in, dtype=np.int32)
    acc = np.ascontiguousarray(accepted, dtype=np.int32)
    g = None if gammas is None else np.ascontiguousarray(gammas, dtype=np.int32)
    B = kv_in.shape[0]
    kv_out = np.zeros(B, dtype=np.int32)
    blocks = np.zeros(B, dtype=np.int32)
    st = np.zeros(B, dtype=np.int32)
    lib().orc_kv_rollback(kv_in.ctypes.data, kv_out.ctypes.data, acc.ctypes.data, _ptr(g),
                          int(gamma_max), B, int(block_size), blocks.ctypes.data, st.ctypes.data)
    return {"kv": kv_out, "blocks": blocks, "status": st}


def accept_terms(w, b: int, i: int, *, draft_tokens=None):
    """(status, p_i(x_i), q_i(x_i)) for sequence b at draft position i."""
    c = _Call(w, draft_tokens=draft_tokens)
    px, qx = ctypes.c_double(), ctypes.c_double()
    st = lib().orc_accept_terms(ctypes.byref(c.args), b, i, ctypes.byref(px), ctypes.byref(qx))
    return st, px.value, qx.value


def position_rows(w, b: int, i: int, *, draft_tokens=None):
    """(status, p_i, q_i, sampling weights, Z) at position i of sequence b."""
    c = _Call(w, draft_tokens=draft_tokens)
    V = w.vocab
    p, q, wt = np.zeros(V), np.zeros(V), np.zeros(V)
    z = ctypes.c_double()
    st = lib().orc_position_rows(ctypes.byref(c.args), b, i, p.ctypes.data, q.ctypes.data,
                                 wt.ctypes.data, ctypes.byref(z))
    return st, p, q, wt, z.value
