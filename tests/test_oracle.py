"""Pins for the fp64 oracle: results fixed by the mathematics, not by the oracle itself.

Each check is chosen so that a plausible slip in ``oracle/kda_oracle.c`` (a
dropped term, a wrong sign or index, a transposed operand, decay applied after
the delta correction, an off-by-one cumulative sum) makes at least one of them
fail; ``test_planted_mistakes_are_caught`` compiles such mutants and proves it.
"""
import math
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kda_d2_t2.txt")


def rand_problem(rng, lens, H, Dk, Dv, with_s0=True, gscale=0.5):
    T = int(sum(lens))
    q = rng.standard_normal((T, H, Dk))
    k = rng.standard_normal((T, H, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, Dv))
    g = -np.abs(rng.standard_normal((T, H, Dk))) * gscale
    beta = rng.uniform(0.05, 1.0, (T, H))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    s0 = rng.standard_normal((len(lens), H, Dk, Dv)) if with_s0 else None
    return q, k, v, g, beta, s0, cu


def forms(orc, chunk=4, seg_len=8):
    """The three oracle forms, each as f(q, k, v, g, beta, scale, s0, cu) -> (out, final)."""
    return {
        "recurrent": lambda *a: orc.recurrent(*a[:6], s0=a[6], cu_seqlens=a[7]),
        "chunked": lambda *a: orc.chunked(*a[:6], s0=a[6], cu_seqlens=a[7], chunk=chunk),
        "segmented": lambda *a: orc.segmented(*a[:6], s0=a[6], cu_seqlens=a[7], chunk=chunk,
                                              seg_len=seg_len),
    }


# --- worked example ------------------------------------------------------------------

def load_golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *nums = line.split()
        vals[key] = np.array([float(x) for x in nums])
    return vals


def golden_check(orc):
    gd = load_golden()
    q = np.stack([gd["q1"], gd["q2"]])[:, None, :]
    k = np.stack([gd["k1"], gd["k2"]])[:, None, :]
    v = np.stack([gd["v1"], gd["v2"]])[:, None, :]
    g = np.log(np.stack([gd["decay1"], gd["decay2"]]))[:, None, :]
    beta = gd["beta"][:, None]
    s0 = gd["s0"].reshape(1, 1, 2, 2)
    exp_out = np.stack([gd["out1"], gd["out2"]])[:, None, :]
    exp_fin = gd["final"].reshape(1, 1, 2, 2)
    res = {}
    for name, f in forms(orc, chunk=2, seg_len=2).items():
        out, fin = f(q, k, v, g, beta, float(gd["scale"][0]), s0, None)
        res[name] = np.allclose(out, exp_out, atol=1e-12) and np.allclose(fin, exp_fin,
                                                                            atol=1e-12)
    for name, f in forms(orc, chunk=1, seg_len=1).items():
        out, fin = f(q, k, v, g, beta, float(gd["scale"][0]), s0, None)
        res[name + "_c1"] = np.allclose(out, exp_out, atol=1e-12) and np.allclose(
            fin, exp_fin, atol=1e-12)
    return res


def test_golden_d2_worked_example(orc):
    res = golden_check(orc)
    assert all(res.values()), res


# --- (a) beta = 0: pure per-channel decay, closed form --------------------------------

def beta_zero_check(orc, rng):
    lens = [21, 1, 40]
    H, D = 2, 6
    q, k, v, g, beta, s0, cu = rand_problem(rng, lens, H, D, D)
    beta[:] = 0.0
    scale = 0.37
    ok = True
    for name, f in forms(orc).items():
        out, fin = f(q, k, v, g, beta, scale, s0, cu)
        for n in range(len(lens)):
            a, b = cu[n], cu[n + 1]
            G = np.cumsum(g[a:b], axis=0)  # [L, H, D]: sum of log-decays up to t
            for h in range(H):
                for t in range(b - a):
                    St = np.exp(G[t, h])[:, None] * s0[n, h]
                    ok &= np.allclose(out[a + t, h], scale * St.T @ q[a + t, h], atol=1e-12)
                Gend = G[-1, h] if b > a else np.zeros(D)
                ok &= np.allclose(fin[n, h], np.exp(Gend)[:, None] * s0[n, h], atol=1e-12)
    return ok


def test_beta_zero_is_pure_decay(orc):
    assert beta_zero_check(orc, np.random.default_rng(11))


# --- (b) beta = 1, unit-norm k: the delta rule stores v_t exactly under k_t -----------

def projection_check(orc, rng, zero_g=False):
    lens = [35, 17]
    H, D = 2, 8
    q, k, v, g, beta, s0, cu = rand_problem(rng, lens, H, D, D)
    if zero_g:
        g[:] = 0.0
    beta[:] = 1.0
    q = k.copy()  # then o_t = scale S_t^T k_t = scale v_t
    scale = 0.61
    ok = True
    for name, f in forms(orc).items():
        out, fin = f(q, k, v, g, beta, scale, s0, cu)
        ok &= np.allclose(out, scale * v, atol=1e-10)
        for n in range(len(lens)):
            t = cu[n + 1] - 1
            for h in range(H):
                ok &= np.allclose(fin[n, h].T @ k[t, h], v[t, h], atol=1e-10)
    return ok


def test_delta_rule_projection_g_zero(orc):
    assert projection_check(orc, np.random.default_rng(12), zero_g=True)


def test_delta_rule_projection_random_g(orc):
    # holds for any g only if the decay is applied before the delta correction
    assert projection_check(orc, np.random.default_rng(13), zero_g=False)


# --- (c) zero state, one token: o = scale * beta * (q . k) * v ------------------------

def single_token_check(orc, rng):
    H, Dk, Dv = 3, 5, 7
    q, k, v, g, beta, _, cu = rand_problem(rng, [1], H, Dk, Dv, with_s0=False)
    k = rng.standard_normal(k.shape)  # any k, not only unit-norm
    scale = 0.29
    ok = True
    for name, f in forms(orc).items():
        out, fin = f(q, k, v, g, beta, scale, None, cu)
        for h in range(H):
            ok &= np.allclose(out[0, h], scale * beta[0, h] * (q[0, h] @ k[0, h]) * v[0, h],
                              atol=1e-13)
            ok &= np.allclose(fin[0, h], beta[0, h] * np.outer(k[0, h], v[0, h]), atol=1e-13)
    return ok


def test_single_token_zero_state(orc):
    assert single_token_check(orc, np.random.default_rng(14))


# --- (d) recurrent vs chunked vs segmented agree to 1e-10 -----------------------------

@pytest.mark.parametrize("T", [1, 15, 16, 17, 33, 100])
@pytest.mark.parametrize("with_s0", [False, True])
def test_forms_agree(orc, T, with_s0):
    rng = np.random.default_rng(100 + T)
    H, D = 2, 16
    q, k, v, g, beta, s0, cu = rand_problem(rng, [T], H, D, D, with_s0=with_s0)
    o1, f1 = orc.recurrent(q, k, v, g, beta, 0.25, s0=s0, cu_seqlens=cu)
    o2, f2 = orc.chunked(q, k, v, g, beta, 0.25, s0=s0, cu_seqlens=cu, chunk=16)
    o3, f3 = orc.segmented(q, k, v, g, beta, 0.25, s0=s0, cu_seqlens=cu, chunk=16, seg_len=32)
    mag = max(1.0, np.abs(o1).max(), np.abs(f1).max())
    for o, f in ((o2, f2), (o3, f3)):
        assert np.abs(o - o1).max() <= 1e-10 * mag
        assert np.abs(f - f1).max() <= 1e-10 * mag


def varlen_agree_check(orc, rng):
    lens = [33, 0, 5, 16, 47]
    H, D = 2, 16
    q, k, v, g, beta, s0, cu = rand_problem(rng, lens, H, D, D)
    o1, f1 = orc.recurrent(q, k, v, g, beta, 0.3, s0=s0, cu_seqlens=cu)
    ok = True
    for chunk, seg in ((16, 32), (4, 8), (16, 16)):
        o2, f2 = orc.chunked(q, k, v, g, beta, 0.3, s0=s0, cu_seqlens=cu, chunk=chunk)
        o3, f3 = orc.segmented(q, k, v, g, beta, 0.3, s0=s0, cu_seqlens=cu, chunk=chunk,
                               seg_len=seg)
        for o, f in ((o2, f2), (o3, f3)):
            ok &= np.abs(o - o1).max() <= 1e-10 and np.abs(f - f1).max() <= 1e-10
    return ok


def test_forms_agree_varlen(orc):
    assert varlen_agree_check(orc, np.random.default_rng(15))


def test_forms_agree_full_head_dim(orc):
    """D = 128 with the configured gate distribution, chunk 16, a ragged tail."""
    rng = np.random.default_rng(16)
    T, H, D = 50, 1, 128
    q = rng.standard_normal((T, H, D))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, D))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, D))
    x = rng.standard_normal((T, H, D))
    g = np.minimum(x, 0) - np.log1p(np.exp(-np.abs(x)))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    s0 = 0.1 * rng.standard_normal((1, H, D, D))
    o1, f1 = orc.recurrent(q, k, v, g, beta, 1 / math.sqrt(D), s0=s0)
    o2, f2 = orc.chunked(q, k, v, g, beta, 1 / math.sqrt(D), s0=s0, chunk=16)
    o3, f3 = orc.segmented(q, k, v, g, beta, 1 / math.sqrt(D), s0=s0, chunk=16, seg_len=32)
    for o, f in ((o2, f2), (o3, f3)):
        assert np.abs(o - o1).max() <= 1e-10
        assert np.abs(f - f1).max() <= 1e-10


# --- extra invariants ------------------------------------------------------------------

def test_linear_in_v_and_state(orc):
    rng = np.random.default_rng(17)
    lens, H, D = [19, 6], 2, 8
    q, k, v1, g, beta, s1, cu = rand_problem(rng, lens, H, D, D)
    v2 = rng.standard_normal(v1.shape)
    s2 = rng.standard_normal(s1.shape)
    a, b = 0.7, -1.3
    for f in forms(orc).values():
        oa, fa = f(q, k, v1, g, beta, 0.5, s1, cu)
        ob, fb = f(q, k, v2, g, beta, 0.5, s2, cu)
        oc, fc = f(q, k, a * v1 + b * v2, g, beta, 0.5, a * s1 + b * s2, cu)
        assert np.allclose(oc, a * oa + b * ob, atol=1e-11)
        assert np.allclose(fc, a * fa + b * fb, atol=1e-11)


def test_sequences_and_heads_independent(orc):
    rng = np.random.default_rng(18)
    lens, H, D = [9, 30, 1], 3, 8
    q, k, v, g, beta, s0, cu = rand_problem(rng, lens, H, D, D)
    out, fin = orc.recurrent(q, k, v, g, beta, 0.4, s0=s0, cu_seqlens=cu)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        for hs in ([0], [2, 1]):
            o, f = orc.chunked(q[a:b][:, hs], k[a:b][:, hs], v[a:b][:, hs], g[a:b][:, hs],
                               beta[a:b][:, hs], 0.4, s0=s0[n:n + 1][:, hs], chunk=16)
            assert np.allclose(o, out[a:b][:, hs], atol=1e-12)
            assert np.allclose(f, fin[n:n + 1][:, hs], atol=1e-12)


def test_continuation_two_calls_equal_one(orc):
    rng = np.random.default_rng(19)
    T, cut, H, D = 45, 21, 2, 8
    q, k, v, g, beta, s0, cu = rand_problem(rng, [T], H, D, D)
    out, fin = orc.recurrent(q, k, v, g, beta, 0.5, s0=s0)
    o1, f1 = orc.chunked(q[:cut], k[:cut], v[:cut], g[:cut], beta[:cut], 0.5, s0=s0, chunk=16)
    o2, f2 = orc.chunked(q[cut:], k[cut:], v[cut:], g[cut:], beta[cut:], 0.5, s0=f1, chunk=16)
    assert np.allclose(np.concatenate([o1, o2]), out, atol=1e-12)
    assert np.allclose(f2, fin, atol=1e-12)


def test_full_forgetting_resets_state(orc):
    """exp(g) = 0 (g = -1e4 in fp64) erases the past: S_t = beta_t k_t v_t^T."""
    rng = np.random.default_rng(20)
    T, H, D = 12, 2, 6
    q, k, v, g, beta, s0, cu = rand_problem(rng, [T], H, D, D)
    g[:] = -1e4
    for f in forms(orc).values():
        out, fin = f(q, k, v, g, beta, 0.5, s0, cu)
        for t in range(T):
            for h in range(H):
                exp_o = 0.5 * beta[t, h] * (q[t, h] @ k[t, h]) * v[t, h]
                assert np.allclose(out[t, h], exp_o, atol=1e-12)
        for h in range(H):
            assert np.allclose(fin[0, h], beta[-1, h] * np.outer(k[-1, h], v[-1, h]),
                               atol=1e-12)


def test_empty_sequences_keep_state(orc):
    rng = np.random.default_rng(21)
    lens, H, D = [0, 4, 0], 2, 4
    q, k, v, g, beta, s0, cu = rand_problem(rng, lens, H, D, D)
    for f in forms(orc).values():
        out, fin = f(q, k, v, g, beta, 0.5, s0, cu)
        assert np.array_equal(fin[0], s0[0]) and np.array_equal(fin[2], s0[2])


def test_invalid_arguments_rejected(orc):
    rng = np.random.default_rng(22)
    q, k, v, g, beta, s0, cu = rand_problem(rng, [4], 1, 4, 4)
    with pytest.raises(ValueError):
        orc.recurrent(q, k, v, g, beta, 1.0, cu_seqlens=np.array([0, 2, 1, 4]))
    with pytest.raises(RuntimeError):
        orc.segmented(q, k, v, g, beta, 1.0, chunk=4, seg_len=6)


# --- the pins catch planted mistakes ----------------------------------------------------

MUTANTS = {
    # delta correction before the decay instead of after it
    "decay_after_delta": (
        r"for \(int64_t i = 0; i < Dk; \+\+i\) \{\n            const double d = exp\(gt\[i\]\);\n"
        r"            for \(int64_t j = 0; j < Dv; \+\+j\) S\[i \* Dv \+ j\] \*= d;\n        \}\n",
        "", "after_update_decay"),
    # o = scale S q instead of scale S^T q
    "output_transposed": (r"ot\[j\] \+= S\[i \* Dv \+ j\] \* qt\[i\];",
                          "ot[j] += S[j * Dv + i] * qt[i];", None),
    # beta dropped from the rank-1 update
    "beta_dropped": (r"u\[j\] = bt \* \(vt\[j\] - u\[j\]\);", "u[j] = (vt[j] - u[j]);", None),
    # prediction uses S k instead of S^T k
    "prediction_transposed": (r"u\[j\] \+= S\[i \* Dv \+ j\] \* kt\[i\];",
                              "u[j] += S[j * Dv + i] * kt[i];", None),
    # chunked: cumulative decay excludes the current row
    "cumsum_off_by_one": (r"acc \+= GROW\(r\)\[i\];\n            w->gam\[r \* Dk \+ i\] = acc;",
                          "w->gam[r * Dk + i] = acc;\n            acc += GROW(r)[i];", None),
    # chunked: wrong sign in the WY forward substitution
    "wy_sign": (r"x -= w->A\[r \* C \+ m\] \* w->T\[m \* C \+ s\];",
                "x += w->A[r * C + m] * w->T[m * C + s];", None),
    # chunked: state decay factor taken at the first row instead of the last
    "chunk_decay_first_row": (r"const double \*glast = w->gam \+ \(C - 1\) \* Dk;\n    for",
                              "const double *glast = w->gam;\n    for", None),
    # segment merge: carry multiplied on the wrong side
    "merge_transposed": (r"acc \+= M\[i \* Dk \+ m\] \* carry\[m \* Dv \+ j\];",
                         "acc += M[m * Dk + i] * carry[m * Dv + j];", None),
}


def _apply_mutant(src, pattern, repl, extra):
    new, n = re.subn(pattern, repl, src, count=1)
    assert n == 1, f"mutation pattern not found: {pattern}"
    if extra == "after_update_decay":
        # re-insert the decay after the rank-1 update
        anchor = "        for (int64_t j = 0; j < Dv; ++j) ot[j] = 0.0;\n"
        decay = ("        for (int64_t i = 0; i < Dk; ++i) {\n"
                 "            const double d = exp(gt[i]);\n"
                 "            for (int64_t j = 0; j < Dv; ++j) S[i * Dv + j] *= d;\n"
                 "        }\n")
        assert anchor in new
        new = new.replace(anchor, decay + anchor, 1)
    return new


def all_pins(orc):
    rng = np.random.default_rng(99)
    results = {
        "golden": all(golden_check(orc).values()),
        "beta_zero": beta_zero_check(orc, rng),
        "projection": projection_check(orc, rng),
        "single_token": single_token_check(orc, rng),
        "varlen_forms": varlen_agree_check(orc, rng),
    }
    return results


def test_pins_pass_on_real_oracle(orc):
    assert all(all_pins(orc).values())


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(tmp_path, name):
    pattern, repl, extra = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    mutated = _apply_mutant(src, pattern, repl, extra)
    cpath = tmp_path / "mutant.c"
    cpath.write_text(mutated)
    so = oracle.build(force=True, src=str(cpath), out=str(tmp_path / "libmutant.so"))
    mut = oracle.OracleLib(so)
    res = all_pins(mut)
    assert not all(res.values()), f"mutant {name} survived every pin: {res}"


@pytest.mark.parametrize("Hq,H", [(2, 6), (6, 2), (3, 3), (1, 4), (4, 1)])
def test_grouped_heads_single_token_closed_form(Hq, H):
    """One token from the zero state: o = scale beta (q . k) v and S = beta k v^T, with
    each output head reading the q, k and state heads the grouping assigns.  Distinct
    values per head make a wrong head map (h * G for h / G, q and k swapped, the state
    of the wrong group member) fail."""
    rng = np.random.default_rng(40 + 7 * Hq + H)
    D = 8
    Hk, Ho = min(Hq, H), max(Hq, H)
    q = rng.standard_normal((1, Hq, D))
    k = rng.standard_normal((1, Hk, D))
    v = rng.standard_normal((1, H, D))
    g = -np.abs(rng.standard_normal((1, H, D)))
    beta = rng.uniform(0.1, 1.0, (1, H))
    scale = 0.37
    out, fin = oracle.grouped(q, k, v, g, beta, scale)
    assert out.shape == (1, Ho, D) and fin.shape == (1, H, D, D)
    for ho in range(Ho):
        if Hq <= H:
            hq = hk = ho // (H // Hq)
            hs = ho
        else:
            hq, hk, hs = ho, ho // (Hq // H), ho // (Hq // H)
        want = scale * beta[0, hs] * np.dot(q[0, hq], k[0, hk]) * v[0, hs]
        np.testing.assert_allclose(out[0, ho], want, rtol=1e-12, atol=1e-12)
    for hs in range(H):
        kk = k[0, hs // (H // Hq)] if Hq <= H else k[0, hs]
        np.testing.assert_allclose(fin[0, hs], beta[0, hs] * np.outer(kk, v[0, hs]),
                                   rtol=1e-12, atol=1e-12)


def test_grouped_heads_equal_counts_is_the_plain_oracle():
    rng = np.random.default_rng(41)
    q, k, v, g, beta, s0, cu = rand_problem(rng, [5, 0, 9], 3, 8, 8)
    a = oracle.grouped(q, k, v, g, beta, 0.3, s0=s0, cu_seqlens=cu)
    b = oracle.recurrent(q, k, v, g, beta, 0.3, s0=s0, cu_seqlens=cu)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
