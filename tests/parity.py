"""Comparison of the CUDA path's outputs with the oracle's, draw by draw.

Rule for the sampling path: tokens, accepted counts and KV lengths must be
identical, except for a mismatching draw whose uniform lies within BAND of
the oracle's decision boundary (|u_acc - p(x)/q(x)| at the first differing
accept test) or of a CDF edge of the emitted token (the oracle's or the
GPU's, under the oracle's weights). Excused mismatches must stay below
1e-4 of all draws; unexcused ones must not occur. A draw is one uniform the
decision consumed: every accept test performed plus the final sample.
"""
from __future__ import annotations

import numpy as np

import oracle
from speculative_decoding_verification_38_gb300 import workloads as wl

BAND = 1e-5
MAX_MISMATCH_FRACTION = 1e-4


def offsets(w):
    if w.target_row_off is not None:
        return np.asarray(w.target_row_off), np.asarray(w.draft_row_off)
    return wl.offsets_for(w.gammas)


class Tally:
    def __init__(self):
        self.draws = 0
        self.mismatches = 0
        self.unexcused = []
        self.in_band = 0
        self.rounds = 0
        self.excused = []  # (kind, distance of u to the boundary)

    def merge(self, o):
        self.draws += o.draws
        self.mismatches += o.mismatches
        self.unexcused += o.unexcused
        self.in_band += o.in_band
        self.rounds += o.rounds
        self.excused += o.excused

    def check(self, label=""):
        assert not self.unexcused, f"{label}: unexcused mismatches {self.unexcused[:10]}"
        assert self.mismatches <= MAX_MISMATCH_FRACTION * self.draws, (
            f"{label}: {self.mismatches} excused mismatches in {self.draws} draws")

    def __repr__(self):
        kinds = {}
        for k, d in self.excused:
            kinds.setdefault(k, []).append(d)
        det = {k: (len(v), float(max(v))) for k, v in kinds.items()}
        return (f"Tally(rounds={self.rounds}, draws={self.draws}, mismatches={self.mismatches}, "
                f"in_band={self.in_band}, unexcused={len(self.unexcused)}, excused(kind: n, max dist)={det})")


def compare_sample(w, gpu: dict, orc: dict, *, seed: int, rnd: int, tokens, seq_offset: int = 0,
                   uniforms=None) -> Tally:
    tro, dro = offsets(w)
    T = Tally()
    T.rounds = 1
    diag = orc["diag"]
    for b in range(w.batch):
        so, sg = orc["status"][b], gpu["status"][b]
        seg = slice(int(tro[b]), int(tro[b + 1]))
        if so != 0 or sg != 0:
            if so != sg or gpu["accepted"][b] != orc["accepted"][b] or \
                    not np.array_equal(gpu["tokens"][seg], orc["tokens"][seg]):
                T.unexcused.append((b, "status", int(so), int(sg)))
            continue
        g = int(dro[b + 1] - dro[b])
        ao, ag = int(orc["accepted"][b]), int(gpu["accepted"][b])
        T.draws += (ao + 1 if ao < g else g) + 1

        def u_of(i):
            if uniforms is not None:
                r = int(tro[b]) + i
                return float(uniforms[r, 0]), float(uniforms[r, 1])
            return oracle.uniform_pair(seed, rnd, seq_offset + b, i)

        band_hit = diag["acc_margin"][b] < BAND or min(abs(diag["u_smp"][b] - diag["cdf_lo"][b]),
                                                         abs(diag["u_smp"][b] - diag["cdf_hi"][b])) < BAND
        T.in_band += int(band_hit)
        same = (ao == ag and np.array_equal(orc["tokens"][seg], gpu["tokens"][seg]))
        if "kv" in orc and same:
            same = orc["kv"][b] == gpu["kv"][b]
            if "blocks" in orc:
                same = same and orc["blocks"][b] == gpu["blocks"][b]
        if same:
            continue
        T.mismatches += 1
        ok = False
        if ao != ag:
            i = min(ao, ag)
            st, px, qx = oracle.accept_terms(w, b, i, draft_tokens=tokens)
            ua, _ = u_of(i)
            ok = st == 0 and qx > 0 and abs(ua - px / qx) < BAND
            if ok:
                T.excused.append(("accept", abs(ua - px / qx)))
        else:
            _, us = u_of(ao)
            dist = min(abs(us - diag["cdf_lo"][b]), abs(us - diag["cdf_hi"][b]))
            ok = dist < BAND
            if not ok:
                tok_g = int(gpu["tokens"][seg][ao])
                if 0 <= tok_g < w.vocab:
                    st, p, q, wts, Z = oracle.position_rows(w, b, ao, draft_tokens=tokens)
                    lo, hi = oracle.cdf_edges(wts, tok_g)
                    dist = min(abs(us - lo), abs(us - hi))
                    ok = dist < BAND
            ok = ok and np.array_equal(orc["tokens"][seg][:ao], gpu["tokens"][seg][:ao])
            if ok:
                T.excused.append(("resid" if ao < g else "bonus", dist))
        if not ok:
            T.unexcused.append((b, ao, ag, orc["tokens"][seg].tolist(), gpu["tokens"][seg].tolist()))
    return T


def compare_exact(w, gpu: dict, orc: dict):
    """Greedy / integer outputs: bit-exact."""
    for k in ("tokens", "accepted", "status", "kv", "blocks"):
        if k in orc:
            assert np.array_equal(gpu[k], orc[k]), (k, np.nonzero(gpu[k] != orc[k])[0][:10])


def compare_tree(w, gpu: dict, orc: dict) -> Tally:
    """Tree verification, sequence by sequence: statuses identical; an OK
    sequence's accepted count, node path and tokens identical, except when
    the oracle's walk met an accept test within BAND of its boundary
    (|u_acc - r(x)/q(x)|, the smallest over the walk) or drew its final
    uniform within BAND of a CDF edge of the emitted token. Draws counted:
    the accepted nodes' tests plus the final draw."""
    T = Tally()
    T.rounds = 1
    diag = orc["diag"]
    off = np.asarray(w.node_off)
    for b in range(w.batch):
        seg = slice(int(off[b]), int(off[b + 1]))
        so, sg = int(orc["status"][b]), int(gpu["status"][b])
        same = (gpu["accepted"][b] == orc["accepted"][b] and np.array_equal(gpu["tokens"][seg], orc["tokens"][seg])
                and np.array_equal(gpu["path"][seg], orc["path"][seg]))
        if so != 0 or sg != 0:
            if so != sg or not same:
                T.unexcused.append((b, "status", so, sg))
            continue
        T.draws += int(orc["accepted"][b]) + 1
        band = diag["acc_margin"][b] < BAND or min(abs(diag["u_smp"][b] - diag["cdf_lo"][b]),
                                                   abs(diag["u_smp"][b] - diag["cdf_hi"][b])) < BAND
        T.in_band += int(band)
        if same:
            continue
        T.mismatches += 1
        if band:
            T.excused.append(("tree", float(min(diag["acc_margin"][b], abs(diag["u_smp"][b] - diag["cdf_lo"][b]),
                                                abs(diag["u_smp"][b] - diag["cdf_hi"][b])))))
        else:
            T.unexcused.append((b, int(orc["accepted"][b]), int(gpu["accepted"][b]), orc["tokens"][seg][:8].tolist(),
                                gpu["tokens"][seg][:8].tolist()))
    return T


# ------------------------------------------------ element-level checks (GPU)
def bulk_copy_path(w, db) -> bool:
    """Whether a sampling call on this batch streams its rows with bulk
    copies: every row starts on a 16-byte boundary (the library's documented
    rule; otherwise the plain-load streaming kernel runs)."""
    esz_t = 2 if w.target.dtype == np.uint16 else 4
    esz_d = 2 if (w.draft is not None and w.draft.dtype == np.uint16) else 4
    ok = (w.vocab * esz_t) % 16 == 0 and db.target.data_ptr() % 16 == 0
    if db.draft is not None:
        ok = ok and (w.vocab * esz_d) % 16 == 0 and db.draft.data_ptr() % 16 == 0
    return ok


def check_debug_probs(sv, w, db, positions, *, same_support=False, tol=1e-5):
    """p_i, q_i, the normalised sampling weights (residual or bonus), p(x),
    q(x) and Z that the GPU path uses, each within tol absolute of the
    oracle's float64 values, for every (sequence, position) listed."""
    import torch

    V = w.vocab
    op, oq, ow = (torch.zeros(V, device="cuda") for _ in range(3))
    sc = torch.zeros(4, device="cuda")
    worst = 0.0
    for b, pos in positions:
        sv.check(sv.spec_debug_probs(db.args, b, pos, op, oq, ow, sc), "debug_probs")
        st, p, q, wts, Z = oracle.position_rows(w, b, pos, draft_tokens=w.draft_tokens)
        assert st == 0
        gp, gq, gw, gs = (t.cpu().numpy().astype(np.float64) for t in (op, oq, ow, sc))
        if same_support:
            assert np.array_equal(gp > 0, p > 0) and np.array_equal(gq > 0, q > 0)
        errs = [np.max(np.abs(gp - p)), np.max(np.abs(gq - q)), np.max(np.abs(gw - wts / wts.sum()))]
        g = int(np.asarray(w.gammas)[b])
        if pos < g:
            _, px, qx = oracle.accept_terms(w, b, pos, draft_tokens=w.draft_tokens)
            errs += [abs(gs[0] - px), abs(gs[1] - qx), abs(gs[2] - Z)]
        worst = max(worst, max(errs))
        assert max(errs) < tol, (b, pos, errs)
    return worst


def check_row_stats(sv, w, db, *, top_ks=None, rel=1e-5):
    """(m, s) of every row against float64: the raw maximum exactly, s =
    sum 2^((l - m) log2(e) / T) (over the columns a top-k keeps) within rel."""
    import torch

    n = w.rows_target + w.rows_draft
    m = torch.zeros(n, device="cuda")
    s = torch.zeros(n, device="cuda")
    sv.check(sv.spec_debug_row_stats(db.args, 0, m, s, None), "row_stats")
    m, s = m.cpu().numpy(), s.cpu().numpy()
    tro, dro = offsets(w)
    L2E = 1.4426950408889634
    temps = np.broadcast_to(np.asarray(w.temperatures if w.temperatures is not None else w.temperature,
                                       dtype=np.float64), (w.batch,))
    worst = 0.0
    for b in range(w.batch):
        T = float(temps[b])
        rows = [(w.target, r, r) for r in range(tro[b], tro[b + 1])] + \
               [(w.draft, r, w.rows_target + r) for r in range(dro[b], dro[b + 1])]
        for arr, r, flat in rows:
            vals = wl.stored_f32(arr[r]).astype(np.float64)
            keep = vals
            if top_ks is not None and 0 < int(top_ks[b]) < vals.size:
                tau = np.sort(vals)[::-1][int(top_ks[b]) - 1]
                keep = vals[vals >= tau]
            assert m[flat] == vals.max()  # the raw maximum, exactly
            ss = np.exp2((keep - vals.max()) / T * L2E).sum()
            worst = max(worst, abs(s[flat] - ss) / ss)
            assert abs(s[flat] - ss) <= rel * ss, (b, r, s[flat], ss)
    return worst
