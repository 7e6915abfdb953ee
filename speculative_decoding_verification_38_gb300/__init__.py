"""Batched speculative-decoding verify on GB300: Python binding of libspecverify.so.

The binding only marshals torch tensors into the C ABI declared in
include/spec_verify.h; every step of the verify runs in the library's CUDA
kernels. There is no CPU fallback: if the shared library is missing or fails
to load, importing the binding's entry points raises.

Low-level entry points (same names as the C ABI):
    spec_verify_workspace_size, spec_workspace_init, spec_verify_sample,
    spec_verify_greedy, spec_kv_rollback, spec_status_string, spec_abi_version,
    spec_debug_philox, spec_debug_row_stats, spec_debug_probs
Convenience: VerifyArgs (builds the argument struct from tensors), Workspace.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_ALIGNMENT = 2
SPEC_ERR_WORKSPACE = 3
SPEC_ERR_CUDA = 4
SPEC_ERR_UNSUPPORTED = 5
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_STATIC_SCRATCH_BYTES = 8 << 20  # scratch of spec_verify_sample_static, per device
SPEC_ABI_VERSION = 5
SEQ_OK, SEQ_BAD_TOKEN, SEQ_BAD_KV, SEQ_BAD_ROW, SEQ_BAD_LAYOUT, SEQ_BAD_TEMP = 0, 1, 2, 3, 4, 5
SEQ_TIMEOUT, SEQ_UNSUPPORTED = 6, 7
SPEC_TREE_MAX_CANDIDATES = 64


class SpecError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {spec_status_string(status)} ({status})")


class SpecVerifyArgs(ctypes.Structure):
    """Mirror of spec_verify_args_t (include/spec_verify.h)."""

    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("batch", ctypes.c_int32),
        ("vocab", ctypes.c_int32),
        ("gamma_max", ctypes.c_int32),
        ("rows_target", ctypes.c_int64),
        ("rows_draft", ctypes.c_int64),
        ("target_row_off", ctypes.c_void_p),
        ("draft_row_off", ctypes.c_void_p),
        ("target_logits", ctypes.c_void_p),
        ("target_dtype", ctypes.c_int32),
        ("draft", ctypes.c_void_p),
        ("draft_dtype", ctypes.c_int32),
        ("draft_is_probs", ctypes.c_int32),
        ("draft_tokens", ctypes.c_void_p),
        ("temperatures", ctypes.c_void_p),
        ("temperature", ctypes.c_float),
        ("seed", ctypes.c_uint64),
        ("round", ctypes.c_uint64),
        ("seq_offset", ctypes.c_uint32),
        ("uniforms", ctypes.c_void_p),
        ("kv_lens_in", ctypes.c_void_p),
        ("kv_lens_out", ctypes.c_void_p),
        ("block_size", ctypes.c_int32),
        ("out_num_blocks", ctypes.c_void_p),
        ("out_tokens", ctypes.c_void_p),
        ("out_accepted", ctypes.c_void_p),
        ("seq_status", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("top_k", ctypes.c_int32),
        ("top_ks", ctypes.c_void_p),
        ("accept_ema", ctypes.c_void_p),
        ("ema_lambda", ctypes.c_float),
        ("top_p", ctypes.c_float),
        ("top_ps", ctypes.c_void_p),
    ]


class SpecTreeArgs(ctypes.Structure):
    """Mirror of spec_tree_args_t (include/spec_verify.h)."""

    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("batch", ctypes.c_int32),
        ("vocab", ctypes.c_int32),
        ("nodes", ctypes.c_int64),
        ("node_off", ctypes.c_void_p),
        ("parent", ctypes.c_void_p),
        ("tokens", ctypes.c_void_p),
        ("target", ctypes.c_void_p),
        ("target_dtype", ctypes.c_int32),
        ("draft", ctypes.c_void_p),
        ("draft_dtype", ctypes.c_int32),
        ("draft_is_probs", ctypes.c_int32),
        ("temperatures", ctypes.c_void_p),
        ("temperature", ctypes.c_float),
        ("seed", ctypes.c_uint64),
        ("round", ctypes.c_uint64),
        ("seq_offset", ctypes.c_uint32),
        ("out_tokens", ctypes.c_void_p),
        ("out_accepted", ctypes.c_void_p),
        ("out_path", ctypes.c_void_p),
        ("seq_status", ctypes.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    from . import buildlib as _b

    return _b.build(force=force)


def lib():
    """The loaded libspecverify.so. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: run "
                                  "`python -c 'import __graft_entry__ as g; g.build()'` first")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, u32, u64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                         ctypes.c_uint64, ctypes.c_size_t)
            A = ctypes.POINTER(SpecVerifyArgs)
            L.spec_abi_version.restype = i32
            L.spec_abi_version.argtypes = []
            L.spec_status_string.restype = ctypes.c_char_p
            L.spec_status_string.argtypes = [ctypes.c_int]
            L.spec_verify_workspace_size.restype = sz
            L.spec_verify_workspace_size.argtypes = [A, i32]
            L.spec_workspace_init.restype = ctypes.c_int
            L.spec_workspace_init.argtypes = [vp, sz, vp]
            L.spec_verify_sample.restype = ctypes.c_int
            L.spec_verify_sample.argtypes = [A, vp]
            L.spec_verify_greedy.restype = ctypes.c_int
            L.spec_verify_greedy.argtypes = [A, vp]
            L.spec_verify_sample_static.restype = ctypes.c_int
            L.spec_verify_sample_static.argtypes = [A, vp]
            L.spec_adapt_gamma.restype = ctypes.c_int
            L.spec_adapt_gamma.argtypes = [vp, i32, i32, ctypes.c_float, i64, vp, vp, vp]
            L.spec_ngram_draft.restype = ctypes.c_int
            L.spec_ngram_draft.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
            L.spec_tree_verify.restype = ctypes.c_int
            L.spec_tree_verify.argtypes = [ctypes.POINTER(SpecTreeArgs), i32, vp]
            L.spec_kv_rollback.restype = ctypes.c_int
            L.spec_kv_rollback.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
            L.spec_debug_philox.restype = ctypes.c_int
            L.spec_debug_philox.argtypes = [u64, u64, u32, i32, i32, vp, vp]
            L.spec_debug_row_stats.restype = ctypes.c_int
            L.spec_debug_row_stats.argtypes = [A, i32, vp, vp, vp, vp]
            L.spec_debug_probs.restype = ctypes.c_int
            L.spec_debug_probs.argtypes = [A, i32, i32, vp, vp, vp, vp, vp]
            L.spec_debug_light_exp2.restype = ctypes.c_int
            L.spec_debug_light_exp2.argtypes = [vp, vp, i64, vp]
            L.spec_debug_time_next_stats.restype = ctypes.c_int
            L.spec_debug_time_next_stats.argtypes = [vp, vp]
            L.spec_debug_set_path.restype = ctypes.c_int
            L.spec_debug_set_path.argtypes = [ctypes.c_int32]
            L.spec_debug_wait_probe.restype = ctypes.c_int
            L.spec_debug_wait_probe.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
            if L.spec_abi_version() != SPEC_ABI_VERSION:
                raise ImportError("libspecverify.so ABI version mismatch")
            _lib = L
    return _lib


# ------------------------------------------------------------------ marshalling
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _check_dev(t, name):
    if t is not None:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


class VerifyArgs:
    """Builds spec_verify_args_t from CUDA tensors and keeps them alive.

    target [rows_target, V] and draft [rows_draft, V] are float32 or bfloat16;
    draft_tokens int32 [rows_draft]; offsets int64 [B+1] (both or neither);
    temperatures float32 [B]; uniforms float32 [rows_target, 2]; kv int32 [B];
    outputs int32. ``workspace`` is a Workspace (or a uint8 CUDA tensor).
    """

    def __init__(self, *, batch, gamma_max, target, draft=None, draft_tokens=None, target_row_off=None,
                 draft_row_off=None, draft_is_probs=False, temperatures=None, temperature=1.0, seed=0, round=0,
                 seq_offset=0, uniforms=None, kv_lens_in=None, kv_lens_out=None, block_size=0,
                 out_num_blocks=None, out_tokens=None, out_accepted=None, seq_status=None, workspace=None,
                 top_k=0, top_ks=None, accept_ema=None, ema_lambda=0.0, top_p=0.0, top_ps=None):
        for name, t in [("target", target), ("draft", draft), ("draft_tokens", draft_tokens), ("top_ks", top_ks),
                        ("accept_ema", accept_ema), ("top_ps", top_ps),
                        ("target_row_off", target_row_off), ("draft_row_off", draft_row_off),
                        ("temperatures", temperatures), ("uniforms", uniforms), ("kv_lens_in", kv_lens_in),
                        ("kv_lens_out", kv_lens_out), ("out_num_blocks", out_num_blocks),
                        ("out_tokens", out_tokens), ("out_accepted", out_accepted), ("seq_status", seq_status)]:
            _check_dev(t, name)
        self.tensors = dict(target=target, draft=draft, draft_tokens=draft_tokens, target_row_off=target_row_off,
                            draft_row_off=draft_row_off, temperatures=temperatures, uniforms=uniforms,
                            kv_lens_in=kv_lens_in, kv_lens_out=kv_lens_out, out_num_blocks=out_num_blocks,
                            out_tokens=out_tokens, out_accepted=out_accepted, seq_status=seq_status,
                            top_ks=top_ks, accept_ema=accept_ema, top_ps=top_ps)
        a = SpecVerifyArgs()
        a.struct_size = ctypes.sizeof(SpecVerifyArgs)
        a.batch = int(batch)
        a.vocab = int(target.shape[1])
        a.gamma_max = int(gamma_max)
        a.rows_target = int(target.shape[0])
        a.rows_draft = int(draft_tokens.shape[0]) if draft_tokens is not None else 0
        a.target_row_off = _ptr(target_row_off)
        a.draft_row_off = _ptr(draft_row_off)
        a.target_logits = _ptr(target)
        a.target_dtype = _dtype_code(target)
        a.draft = _ptr(draft)
        a.draft_dtype = _dtype_code(draft) if draft is not None else SPEC_F32
        a.draft_is_probs = int(bool(draft_is_probs))
        a.draft_tokens = _ptr(draft_tokens)
        a.temperatures = _ptr(temperatures)
        a.temperature = float(temperature)
        a.seed = int(seed)
        a.round = int(round)
        a.seq_offset = int(seq_offset)
        a.uniforms = _ptr(uniforms)
        a.kv_lens_in = _ptr(kv_lens_in)
        a.kv_lens_out = _ptr(kv_lens_out)
        a.block_size = int(block_size)
        a.out_num_blocks = _ptr(out_num_blocks)
        a.out_tokens = _ptr(out_tokens)
        a.out_accepted = _ptr(out_accepted)
        a.seq_status = _ptr(seq_status)
        a.top_k = int(top_k)
        a.top_ks = _ptr(top_ks)
        a.accept_ema = _ptr(accept_ema)
        a.ema_lambda = float(ema_lambda)
        a.top_p = float(top_p)
        a.top_ps = _ptr(top_ps)
        self.struct = a
        self.workspace = None
        if workspace is not None:
            self.set_workspace(workspace)

    def set_workspace(self, ws):
        buf = ws.buffer if isinstance(ws, Workspace) else ws
        self.workspace = ws
        self.struct.workspace = buf.data_ptr()
        self.struct.workspace_bytes = buf.numel() * buf.element_size()

    def set_round(self, rnd: int):
        self.struct.round = int(rnd)

    def set_top_k(self, top_k=0, top_ks=None):
        """Top-k truncation of every row (k <= 0 or k >= V: off); top_ks int32 [B] per sequence."""
        _check_dev(top_ks, "top_ks")
        self.tensors["top_ks"] = top_ks
        self.struct.top_k = int(top_k)
        self.struct.top_ks = _ptr(top_ks)

    def set_accept_ema(self, accept_ema=None, ema_lambda=0.0):
        """Running acceptance (float32 [B], updated in place by each verify call) or None."""
        _check_dev(accept_ema, "accept_ema")
        self.tensors["accept_ema"] = accept_ema
        self.struct.accept_ema = _ptr(accept_ema)
        self.struct.ema_lambda = float(ema_lambda)

    def set_tokens(self, draft_tokens):
        _check_dev(draft_tokens, "draft_tokens")
        self.tensors["draft_tokens"] = draft_tokens
        self.struct.draft_tokens = _ptr(draft_tokens)


class Workspace:
    """A caller-owned device workspace (uint8 CUDA tensor), initialised once."""

    def __init__(self, nbytes: int, device=None, stream=None):
        import torch

        nbytes = max(int(nbytes), 1)
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
        check(spec_workspace_init(self.buffer.data_ptr(), nbytes, stream), "spec_workspace_init")

    @classmethod
    def for_args(cls, args: VerifyArgs, greedy: bool, device=None, stream=None, slack: float = 1.0):
        n = spec_verify_workspace_size(args, greedy)
        if n == 0:
            raise SpecError(SPEC_ERR_INVALID_ARG, "spec_verify_workspace_size")
        return cls(int(n * slack), device=device, stream=stream)


def check(status: int, what: str = "spec call"):
    if status != SPEC_OK:
        raise SpecError(status, what)
    return status


# ------------------------------------------------------------- C ABI wrappers
def spec_abi_version() -> int:
    return lib().spec_abi_version()


def spec_status_string(status: int) -> str:
    try:
        return lib().spec_status_string(int(status)).decode()
    except ImportError:
        return f"status {status}"


def spec_verify_workspace_size(args: VerifyArgs, greedy: bool) -> int:
    return int(lib().spec_verify_workspace_size(ctypes.byref(args.struct), int(bool(greedy))))


def spec_workspace_init(ptr: int, nbytes: int, stream=None) -> int:
    return lib().spec_workspace_init(ptr, nbytes, _stream(stream))


def spec_verify_sample(args: VerifyArgs, stream=None) -> int:
    return lib().spec_verify_sample(ctypes.byref(args.struct), _stream(stream))


def spec_adapt_gamma(accept_ema, gamma_max: int, draft_cost: float, gammas_out, max_positions: int = 0,
                     total_positions_out=None, stream=None) -> int:
    """Next-round gamma per request from the running acceptance (all device tensors)."""
    for name, t in [("accept_ema", accept_ema), ("gammas_out", gammas_out), ("total_positions_out", total_positions_out)]:
        _check_dev(t, name)
    return lib().spec_adapt_gamma(accept_ema.data_ptr(), int(accept_ema.numel()), int(gamma_max), float(draft_cost),
                                  int(max_positions), gammas_out.data_ptr(), _ptr(total_positions_out), _stream(stream))


def spec_ngram_draft(ctx, ctx_off, n_max: int, n_min: int, gamma: int, draft_out, n_draft_out, match_pos_out=None,
                     match_n_out=None, stream=None) -> int:
    """Prompt-lookup drafts for every sequence (all device tensors; ctx int32, ctx_off int64 [B+1])."""
    for name, t in [("ctx", ctx), ("ctx_off", ctx_off), ("draft_out", draft_out), ("n_draft_out", n_draft_out),
                    ("match_pos_out", match_pos_out), ("match_n_out", match_n_out)]:
        _check_dev(t, name)
    return lib().spec_ngram_draft(_ptr(ctx) if ctx is not None and ctx.numel() else None, ctx_off.data_ptr(),
                                  int(ctx_off.numel() - 1), int(n_max), int(n_min), int(gamma), draft_out.data_ptr(),
                                  n_draft_out.data_ptr(), _ptr(match_pos_out), _ptr(match_n_out), _stream(stream))


def tree_args(*, node_off, parent, tokens, target, draft=None, draft_is_probs=False, temperatures=None,
              temperature=1.0, seed=0, rnd=0, seq_offset=0, out_tokens, out_accepted, out_path=None,
              seq_status=None) -> SpecTreeArgs:
    """spec_tree_args_t over device tensors: node_off int64 [B+1]; parent,
    tokens int32 [nodes]; target (and draft) [nodes, V] float32 or bfloat16."""
    for name, t in [("node_off", node_off), ("parent", parent), ("tokens", tokens), ("target", target),
                    ("draft", draft), ("temperatures", temperatures), ("out_tokens", out_tokens),
                    ("out_accepted", out_accepted), ("out_path", out_path), ("seq_status", seq_status)]:
        _check_dev(t, name)
    a = SpecTreeArgs()
    a.struct_size = ctypes.sizeof(SpecTreeArgs)
    a.batch = int(node_off.numel() - 1)
    a.vocab = int(target.shape[1])
    a.nodes = int(target.shape[0])
    a.node_off, a.parent, a.tokens = node_off.data_ptr(), parent.data_ptr(), tokens.data_ptr()
    a.target, a.target_dtype = target.data_ptr(), _dtype_code(target)
    if draft is not None:
        a.draft, a.draft_dtype = draft.data_ptr(), _dtype_code(draft)
    a.draft_is_probs = int(bool(draft_is_probs))
    a.temperatures = _ptr(temperatures)
    a.temperature = float(temperature)
    a.seed, a.round, a.seq_offset = int(seed) & (2**64 - 1), int(rnd) & (2**64 - 1), int(seq_offset)
    a.out_tokens, a.out_accepted = out_tokens.data_ptr(), out_accepted.data_ptr()
    a.out_path, a.seq_status = _ptr(out_path), _ptr(seq_status)
    return a


def spec_tree_verify(args: SpecTreeArgs, greedy: bool = False, stream=None) -> int:
    """Verify every sequence's token tree in one launch (see tree_args)."""
    return lib().spec_tree_verify(ctypes.byref(args), int(bool(greedy)), _stream(stream))


def spec_verify_greedy(args: VerifyArgs, stream=None) -> int:
    return lib().spec_verify_greedy(ctypes.byref(args.struct), _stream(stream))


def spec_verify_sample_static(args: VerifyArgs, stream=None) -> int:
    """spec_verify_sample on the library's own fixed scratch (8 MiB per device)
    for callers that cannot provide device memory; args' workspace is ignored.
    Calls that overlap on the GPU race on that scratch."""
    return lib().spec_verify_sample_static(ctypes.byref(args.struct), _stream(stream))


def spec_kv_rollback(kv_in, kv_out, accepted, gammas, gamma_max, block_size=0, out_num_blocks=None,
                     seq_status=None, stream=None) -> int:
    for name, t in [("kv_in", kv_in), ("kv_out", kv_out), ("accepted", accepted), ("gammas", gammas),
                    ("out_num_blocks", out_num_blocks), ("seq_status", seq_status)]:
        _check_dev(t, name)
    return lib().spec_kv_rollback(_ptr(kv_in), _ptr(kv_out), _ptr(accepted), _ptr(gammas), int(gamma_max),
                                  int(kv_in.shape[0]), int(block_size), _ptr(out_num_blocks), _ptr(seq_status),
                                  _stream(stream))


def spec_debug_philox(seed, rnd, seq_offset, batch, npos, out, stream=None) -> int:
    _check_dev(out, "out")
    return lib().spec_debug_philox(int(seed), int(rnd), int(seq_offset), int(batch), int(npos), _ptr(out),
                                   _stream(stream))


def spec_debug_row_stats(args: VerifyArgs, greedy, out_a=None, out_b=None, out_idx=None, stream=None) -> int:
    return lib().spec_debug_row_stats(ctypes.byref(args.struct), int(bool(greedy)), _ptr(out_a), _ptr(out_b),
                                      _ptr(out_idx), _stream(stream))


def spec_debug_probs(args: VerifyArgs, seq, pos, out_p=None, out_q=None, out_w=None, out_scalars=None,
                     stream=None) -> int:
    return lib().spec_debug_probs(ctypes.byref(args.struct), int(seq), int(pos), _ptr(out_p), _ptr(out_q),
                                  _ptr(out_w), _ptr(out_scalars), _stream(stream))


def spec_debug_time_next_stats(start_event=None, stop_event=None) -> int:
    """Arm the hook: the next verify call on this thread records the two torch
    CUDA events around its streaming pass."""
    a = None if start_event is None else start_event.cuda_event
    b = None if stop_event is None else stop_event.cuda_event
    return lib().spec_debug_time_next_stats(a, b)


PATH_DEFAULT, PATH_SEPARATE, PATH_FUSED = 0, 1, 2


def spec_debug_set_path(path: int) -> int:
    """Process-wide test switch for sampling calls: PATH_DEFAULT, PATH_SEPARATE
    (the streaming, finalize, tile and draw kernels) or PATH_FUSED (the one
    cooperative kernel, wherever it applies)."""
    return lib().spec_debug_set_path(int(path))


def spec_debug_wait_probe(flag, limit_ns: int, out, stream=None) -> int:
    """One warp's bounded wait on the device word flag[0] (the fused kernel's
    hand-off wait): out[0] = the value seen (0 if it gave up), out[1] = 1 if
    it gave up. flag and out: uint32 (or int32) CUDA tensors."""
    return lib().spec_debug_wait_probe(flag.data_ptr(), int(limit_ns), out.data_ptr(), _stream(stream))


def spec_debug_light_exp2(x, y, stream=None) -> int:
    """The sampler's light-weight 2^x for every element of x, as (value,
    correction) pairs in y (float32 CUDA tensors, y has 2 * len(x) entries)."""
    _check_dev(x, "x")
    _check_dev(y, "y")
    return lib().spec_debug_light_exp2(_ptr(x), _ptr(y), int(x.numel()), _stream(stream))
