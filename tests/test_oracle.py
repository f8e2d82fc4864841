"""The fp64 oracle against closed forms, invariants, dense expansions and
exact rationals; and proof that those pins catch plausible mistakes."""
import os

import numpy as np
import pytest

import oracle
import pins
from oracle import chunk_model


@pytest.mark.parametrize("name", sorted(pins.ALL_CHECKS))
def test_pin(oracle_lib, name):
    fn, tol = pins.ALL_CHECKS[name]
    err = fn(oracle_lib)
    assert err <= tol, f"{name}: rel err {err:.3e} > {tol:.1e}"


# Plausible mistakes, planted in a copy of the oracle source (on the CPU).
# Each must make at least one pin fail.
MUTANTS = {
    "drop_decay_in_correction": ("v[i] - a * x", "v[i] - x"),
    "wrong_sign_rank1": ("row[j] = a * row[j] + u * k[j]", "row[j] = a * row[j] - u * k[j]"),
    "beta_only_on_value": ("beta * (v[i] - a * x)", "(beta * v[i] - a * x)"),
    "output_from_old_state": ("y += row[j] * q[j]", "y += (row[j] - u * k[j]) * q[j]"),
    "query_is_key": ("y += row[j] * q[j]", "y += row[j] * k[j]"),
    "gqa_interleaved": ("const int64_t hk = h / group;\n        double *S",
                        "const int64_t hk = h % Hk;\n        double *S"),
    "decode_gqa_interleaved": ("const int64_t hk = h / group;\n        gdn_token_step",
                               "const int64_t hk = h % Hk;\n        gdn_token_step"),
    "decay_squared": ("const double a = exp(g);", "const double a = exp(2.0 * g);"),
    "drop_last_token": ("t < cu_seqlens[n + 1]; ++t", "t + 1 < cu_seqlens[n + 1]; ++t"),
    "ignore_initial_state": ("if (initial_state)\n", "if (0)\n"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(path), out=str(tmp_path / f"lib{name}.so"), force=True))
    failed = []
    for pname, (fn, tol) in pins.ALL_CHECKS.items():
        try:
            err = fn(lib)
        except Exception:
            err = np.inf
        if not (err <= tol):
            failed.append(pname)
    assert failed, f"mutant {name} passed every pin"


def _random_problem(rng, lens, Hk, Hv, d, h0=True):
    T = sum(lens)
    q = pins.unit(rng.standard_normal((T, Hk, d)))
    k = pins.unit(rng.standard_normal((T, Hk, d)))
    v = rng.standard_normal((T, Hv, d))
    g = -0.1 * np.logaddexp(0, rng.standard_normal((T, Hv)))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, Hv))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S0 = 0.5 * rng.standard_normal((len(lens), Hv, d, d)) if h0 else None
    return q, k, v, g, b, cu, S0


@pytest.mark.parametrize("chunk", [1, 2, 3, 16, 64])
def test_chunk_model_matches_oracle(oracle_lib, chunk):
    """The chunked (WY/UT) algebra the kernels use equals the token recurrence."""
    rng = np.random.default_rng(10 + chunk)
    q, k, v, g, b, cu, S0 = _random_problem(rng, [70, 0, 5, 130], 2, 4, 8)
    o_ref, f_ref = oracle.prefill(q, k, v, g, b, cu, S0, lib=oracle_lib)
    o, f = chunk_model.prefill(q, k, v, g, b, cu, S0, chunk=chunk)
    assert pins.rel(o, o_ref) <= 1e-12
    assert pins.rel(f, f_ref) <= 1e-12


def test_varlen_equals_separate_runs(oracle_lib):
    rng = np.random.default_rng(20)
    lens = [3, 0, 17, 9]
    q, k, v, g, b, cu, S0 = _random_problem(rng, lens, 1, 3, 6)
    out, fin = oracle.prefill(q, k, v, g, b, cu, S0, lib=oracle_lib)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        o1, f1 = oracle.prefill(q[s:e], k[s:e], v[s:e], g[s:e], b[s:e], [0, e - s],
                                S0[n:n + 1], lib=oracle_lib)
        assert np.array_equal(o1, out[s:e])
        assert np.array_equal(f1[0], fin[n])


def test_split_prefill_equals_whole(oracle_lib):
    """prefill(T1) then prefill(T2) from its final state == prefill(T1 + T2)."""
    rng = np.random.default_rng(21)
    q, k, v, g, b, cu, S0 = _random_problem(rng, [40], 2, 2, 5)
    out, fin = oracle.prefill(q, k, v, g, b, cu, S0, lib=oracle_lib)
    o1, f1 = oracle.prefill(q[:13], k[:13], v[:13], g[:13], b[:13], [0, 13], S0, lib=oracle_lib)
    o2, f2 = oracle.prefill(q[13:], k[13:], v[13:], g[13:], b[13:], [0, 27], f1, lib=oracle_lib)
    assert np.array_equal(np.concatenate([o1, o2]), out)
    assert np.array_equal(f2, fin)


def test_head_subset_matches_full(oracle_lib):
    rng = np.random.default_rng(22)
    q, k, v, g, b, cu, S0 = _random_problem(rng, [12, 7], 2, 6, 4)
    out, fin = oracle.prefill(q, k, v, g, b, cu, S0, lib=oracle_lib)
    heads = [1, 4, 5]
    o2, f2 = oracle.prefill(q, k, v, g, b, cu, S0, heads=heads, lib=oracle_lib)
    assert np.array_equal(o2[:, heads], out[:, heads])
    assert np.isnan(o2[:, [0, 2, 3]]).all()
    assert np.array_equal(f2[:, heads], fin[:, heads])


def test_state_norm_bound(oracle_lib):
    """With unit keys and b in [0, 1], I - b k k^T has spectral norm <= 1, so
    ||S_t||_F <= a_t ||S_{t-1}||_F + b_t ||v_t||."""
    rng = np.random.default_rng(23)
    T, d = 50, 7
    q, k, v, g, b, cu, S0 = _random_problem(rng, [T], 1, 1, d)
    prev = np.linalg.norm(S0[0, 0])
    for t in range(T):
        _, f = oracle.prefill(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1], b[:t + 1],
                              [0, t + 1], S0, lib=oracle_lib)
        cur = np.linalg.norm(f[0, 0])
        bound = np.exp(g[t, 0]) * prev + b[t, 0] * np.linalg.norm(v[t, 0])
        assert cur <= bound * (1 + 1e-12)
        prev = cur


def test_thread_count_does_not_change_results(oracle_lib):
    rng = np.random.default_rng(24)
    q, k, v, g, b, cu, S0 = _random_problem(rng, [33, 21], 2, 4, 6)
    o1, f1 = oracle.prefill(q, k, v, g, b, cu, S0, num_threads=1, lib=oracle_lib)
    o2, f2 = oracle.prefill(q, k, v, g, b, cu, S0, num_threads=3, lib=oracle_lib)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_rejects_bad_head_grouping(oracle_lib):
    z = np.zeros((2, 2, 3))
    with pytest.raises(ValueError):
        oracle.prefill(z, z, np.zeros((2, 3, 3)), np.zeros((2, 3)), np.zeros((2, 3)), [0, 2],
                       lib=oracle_lib)
