"""Host-side checks of the C ABI (no GPU): the library builds, loads, exports
every symbol include/spec_verify.h declares, its struct layout matches the
binding, and host validation rejects bad arguments before any CUDA call."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_38_gb300 as sv

    sv.build()
    return sv


def declared_symbols():
    src = open(HEADER).read()
    return re.findall(r"SPEC_API\s+[\w\s\*]+?\b(spec_\w+)\s*\(", src)


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ["spec_verify_sample", "spec_verify_greedy", "spec_kv_rollback", "spec_verify_workspace_size",
              "spec_workspace_init", "spec_status_string", "spec_abi_version"]:
        assert s in syms


def test_library_exports_every_declared_symbol(sv):
    L = sv.lib()
    for s in declared_symbols():
        assert hasattr(L, s), s
    nm = subprocess.run(["nm", "-D", "--defined-only", sv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\s[TW]\s(\w+)$", nm, re.M))
    spec_exports = {e for e in exported if e.startswith("spec_")}
    assert spec_exports == set(declared_symbols())


@pytest.mark.parametrize("cname,pyname", [("spec_verify_args_t", "SpecVerifyArgs"),
                                           ("spec_tree_args_t", "SpecTreeArgs")])
def test_struct_layout_matches_header(sv, cname, pyname):
    S = getattr(sv, pyname)
    fields = [f for f, _ in S._fields_]
    prog = "#include <stdio.h>\n#include <stddef.h>\n#include \"spec_verify.h\"\nint main(void){\n"
    prog += f'printf("%zu\\n", sizeof({cname}));\n'
    for f in fields:
        prog += f'printf("%zu\\n", offsetof({cname}, {f}));\n'
    prog += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(prog)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        out = [int(x) for x in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(S)
    assert len(out) == len(fields) + 1
    for f, off in zip(fields, out[1:]):
        assert getattr(S, f).offset == off, f


def test_abi_version_and_status_strings(sv):
    assert sv.spec_abi_version() == 5 == sv.SPEC_ABI_VERSION
    assert sv.spec_status_string(0) == "SPEC_OK"
    assert sv.spec_status_string(3) == "SPEC_ERR_WORKSPACE"


def _args(sv, **kw):
    a = sv.SpecVerifyArgs()
    a.struct_size = ctypes.sizeof(sv.SpecVerifyArgs)
    a.batch, a.vocab, a.gamma_max = kw.get("batch", 4), kw.get("vocab", 1000), kw.get("gamma", 3)
    a.rows_target = kw.get("rows_target", a.batch * (a.gamma_max + 1))
    a.rows_draft = kw.get("rows_draft", a.batch * a.gamma_max)
    fake = 1 << 20  # never dereferenced: validation fails before any launch
    a.target_logits = kw.get("target", fake)
    a.draft = kw.get("draft", fake)
    a.draft_tokens = kw.get("tokens", fake)
    a.out_tokens = kw.get("out_tokens", fake)
    a.out_accepted = fake
    a.temperature = kw.get("temperature", 1.0)
    a.workspace = kw.get("workspace", fake)
    a.workspace_bytes = 1 << 30
    a.target_dtype = kw.get("tdt", 1)
    a.draft_dtype = 1
    return a


def test_workspace_size_is_host_arithmetic(sv):
    L = sv.lib()
    a = _args(sv)
    n = L.spec_verify_workspace_size(ctypes.byref(a), 0)
    assert n > 0 and n % 256 == 0
    big = _args(sv, batch=64, gamma=8, vocab=128256)
    assert L.spec_verify_workspace_size(ctypes.byref(big), 0) >= L.spec_verify_workspace_size(ctypes.byref(big), 1)
    bad = _args(sv, rows_target=7)  # uniform layout needs B*(gamma+1) rows
    assert L.spec_verify_workspace_size(ctypes.byref(bad), 0) == 0
    assert L.spec_verify_workspace_size(None, 0) == 0


def test_workspace_grows_by_4kb_per_row_when_top_p_may_be_asked(sv):
    L = sv.lib()
    for top_p, top_ps in ((0.9, None), (0.0, 1 << 20)):
        plain, topp = _args(sv, batch=64, gamma=8, vocab=128256), _args(sv, batch=64, gamma=8, vocab=128256)
        topp.top_p = top_p
        if top_ps:
            topp.top_ps = top_ps
        rows = plain.rows_target + plain.rows_draft
        n0, n1 = (L.spec_verify_workspace_size(ctypes.byref(x), 0) for x in (plain, topp))
        assert n1 - n0 >= rows * 4096 and n1 - n0 < rows * 4096 + rows * 4 + 512
        # greedy ignores top-p
        assert L.spec_verify_workspace_size(ctypes.byref(topp), 1) == L.spec_verify_workspace_size(
            ctypes.byref(plain), 1)
    off = _args(sv, batch=64, gamma=8, vocab=128256)
    off.top_p = 1.0  # top-p off: no extra room
    assert L.spec_verify_workspace_size(ctypes.byref(off), 0) == L.spec_verify_workspace_size(
        ctypes.byref(_args(sv, batch=64, gamma=8, vocab=128256)), 0)


def test_host_validation_rejects_before_cuda(sv):
    L = sv.lib()

    def call(a, greedy=False):
        f = L.spec_verify_greedy if greedy else L.spec_verify_sample
        return f(ctypes.byref(a), None)

    assert L.spec_verify_sample(None, None) == sv.SPEC_ERR_INVALID_ARG
    a = _args(sv)
    a.struct_size = 8
    assert call(a) == sv.SPEC_ERR_INVALID_ARG
    assert call(_args(sv, batch=0)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_args(sv, gamma=65)) == sv.SPEC_ERR_UNSUPPORTED
    assert call(_args(sv, target=0)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_args(sv, target=(1 << 20) + 1)) == sv.SPEC_ERR_ALIGNMENT
    assert call(_args(sv, temperature=0.0)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_args(sv, temperature=float("nan"))) == sv.SPEC_ERR_INVALID_ARG
    assert call(_args(sv, workspace=(1 << 20) + 16)) == sv.SPEC_ERR_WORKSPACE
    assert call(_args(sv, workspace=0)) == sv.SPEC_ERR_WORKSPACE
    assert call(_args(sv, tdt=7)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_args(sv, tdt=7), greedy=True) == sv.SPEC_ERR_INVALID_ARG
    a = _args(sv)
    a.top_ks = (1 << 20) + 2  # per-sequence k must be int32-aligned
    assert call(a) == sv.SPEC_ERR_ALIGNMENT
    a = _args(sv)
    a.top_ps = (1 << 20) + 2  # per-sequence p must be float32-aligned
    assert call(a) == sv.SPEC_ERR_ALIGNMENT
    # the struct grew with top_k / top_ks: the size of the previous layout is rejected
    a = _args(sv)
    a.struct_size = sv.SpecVerifyArgs.top_k.offset
    assert call(a) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_kv_rollback(None, None, None, None, 3, 4, 0, None, None, None) == sv.SPEC_ERR_INVALID_ARG
    fake = 1 << 20
    assert L.spec_adapt_gamma(None, 4, 8, 0.05, 0, fake, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_adapt_gamma(fake, 0, 8, 0.05, 0, fake, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_adapt_gamma(fake, 4, 65, 0.05, 0, fake, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_adapt_gamma(fake, 4, 8, float("nan"), 0, fake, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_adapt_gamma(fake + 2, 4, 8, 0.05, 0, fake, None, None) == sv.SPEC_ERR_ALIGNMENT
    ng = L.spec_ngram_draft
    assert ng(fake, None, 4, 3, 1, 8, fake, fake, None, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert ng(fake, fake, 4, 3, 0, 8, fake, fake, None, None, None) == sv.SPEC_ERR_INVALID_ARG  # n_min < 1
    assert ng(fake, fake, 4, 2, 3, 8, fake, fake, None, None, None) == sv.SPEC_ERR_INVALID_ARG  # n_max < n_min
    assert ng(fake, fake, 4, 17, 1, 8, fake, fake, None, None, None) == sv.SPEC_ERR_INVALID_ARG  # n_max > 16
    assert ng(fake, fake, 4, 3, 1, 65, fake, fake, None, None, None) == sv.SPEC_ERR_INVALID_ARG  # gamma > 64
    assert ng(fake, fake + 4, 4, 3, 1, 8, fake, fake, None, None, None) == sv.SPEC_ERR_ALIGNMENT  # ctx_off int64
    a = _args(sv)
    a.accept_ema = fake
    a.ema_lambda = 1.5  # outside [0, 1]
    assert call(a) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_debug_philox(0, 0, 0, 0, 1, None, None) == sv.SPEC_ERR_INVALID_ARG


def _tree_args(sv, **kw):
    fake = 1 << 20  # never dereferenced: validation fails before any launch
    a = sv.SpecTreeArgs()
    a.struct_size = ctypes.sizeof(sv.SpecTreeArgs)
    a.batch, a.vocab, a.nodes = kw.get("batch", 4), kw.get("vocab", 1000), kw.get("nodes", 28)
    a.node_off, a.parent, a.tokens = kw.get("node_off", fake), fake, fake
    a.target, a.target_dtype = kw.get("target", fake), kw.get("tdt", 1)
    a.draft, a.draft_dtype, a.draft_is_probs = kw.get("draft", fake), 1, kw.get("probs", 0)
    a.temperature = 1.0
    a.out_tokens, a.out_accepted = fake, fake
    a.out_path = kw.get("out_path", None)
    return a


def test_tree_host_validation(sv):
    L = sv.lib()

    def call(a, greedy=0):
        return L.spec_tree_verify(ctypes.byref(a), greedy, None)

    assert L.spec_tree_verify(None, 0, None) == sv.SPEC_ERR_INVALID_ARG
    a = _tree_args(sv)
    a.struct_size = 8
    assert call(a) == sv.SPEC_ERR_INVALID_ARG
    assert call(_tree_args(sv, batch=0)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_tree_args(sv, vocab=0)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_tree_args(sv, vocab=(1 << 21) + 1)) == sv.SPEC_ERR_UNSUPPORTED
    assert call(_tree_args(sv, nodes=3)) == sv.SPEC_ERR_INVALID_ARG  # fewer nodes than sequences
    assert call(_tree_args(sv, nodes=1 << 31)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_tree_args(sv, target=0)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_tree_args(sv, tdt=3)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_tree_args(sv, draft=0)) == sv.SPEC_ERR_INVALID_ARG  # sampling reads draft rows
    assert call(_tree_args(sv, probs=2)) == sv.SPEC_ERR_INVALID_ARG
    assert call(_tree_args(sv, node_off=(1 << 20) + 4)) == sv.SPEC_ERR_ALIGNMENT
    assert call(_tree_args(sv, target=(1 << 20) + 1)) == sv.SPEC_ERR_ALIGNMENT
    assert call(_tree_args(sv, out_path=(1 << 20) + 2)) == sv.SPEC_ERR_ALIGNMENT


def test_binding_fails_loudly_without_library(sv, tmp_path, monkeypatch):
    import speculative_decoding_verification_38_gb300 as pkg

    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        pkg.lib()
