"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Every mutant is a textual substitution in oracle/gdn_oracle.c (applied to a copy in a
temporary directory, compiled with the oracle's own gcc flags). The test fails if a
substitution no longer matches the source (the list went stale) or if a mutant passes
every pin in tests/oracle_pins.py.
"""
import os

import pytest

import oracle
import oracle_pins as P

# (name, old text, new text, expected number of matches)
MUTANTS = [
    ("readout adjoint dropped", "+= dyt[i] * qt[j];", "+= 0.0 * dyt[i] * qt[j];", 1),
    ("readout adjoint uses k", "+= dyt[i] * qt[j];", "+= dyt[i] * kt[j];", 1),
    ("sign of du", "du[i] = -bt * dd[i];", "du[i] = bt * dd[i];", 1),
    ("dg reads S_t", "dgt += dA[e] * Sprev[e];", "dgt += dA[e] * Scur[e];", 1),
    ("GQA head index modulo", "hk = h / rep", "hk = h % s->Hk", 2),
    ("A^T du misses g", "acc += (gt * Sprev[(size_t)i * Dk + j]) * du[i];",
     "acc += (Sprev[(size_t)i * Dk + j]) * du[i];", 1),
    ("A^T du dropped", "acc += (gt * Sprev[(size_t)i * Dk + j]) * du[i];", "acc += 0.0 * du[i];", 1),
    ("prediction before decay", "acc += S[(size_t)i * Dk + j] * kt[j];  /* u = S k */",
     "acc += S[(size_t)i * Dk + j] / gt * kt[j];", 1),
    ("readout before write", "acc += S[(size_t)i * Dk + j] * qt[j];  /* y = S q */",
     "acc += (S[(size_t)i * Dk + j] - delta[i] * kt[j]) * qt[j];", 1),
    ("dq reads S_{t-1}", "acc += Scur[(size_t)i * Dk + j] * dyt[i];",
     "acc += Sprev[(size_t)i * Dk + j] * dyt[i];", 1),
    ("Sh^T delta uses ddelta", "acc += Sh[(size_t)i * Dk + j] * delta[i];",
     "acc += Sh[(size_t)i * Dk + j] * dd[i];", 1),
    ("carry without decay", "Sh[e] = gt * dA[e];", "Sh[e] = dA[e];", 1),
    ("dbeta ignores prediction", "db += dd[i] * (vt[i] - u[i]);", "db += dd[i] * vt[i];", 1),
    ("dv misses beta", "dv[off_v(s, b, t, h) + i] = bt * dd[i];", "dv[off_v(s, b, t, h) + i] = dd[i];", 1),
    ("forward drops beta", "delta[i] = bt * (vt[i] - u[i]);", "delta[i] = (vt[i] - u[i]);", 1),
    ("dA misses du k^T", "+ du[i] * kt[j];", "+ 0.0 * du[i] * kt[j];", 1),
]

# quick pins first: a mutant is killed by the first pin that fails
ORDER = [P.pin_single_step, P.pin_zero_decay, P.pin_identity_decay_no_write, P.pin_exact_retrieval,
         P.pin_fixed_unit_key, P.pin_orthonormal_keys, P.pin_dot_product, P.pin_directional_fd,
         P.pin_forward_mode_jacobian, P.pin_finite_differences, P.pin_strong_decay_dot_product]

# mistakes in how the decay enters; the strong-decay pin (g in [1e-4, 1e-3]) must catch each
# on its own, so that the regime where chunked kernels have lost dg stays covered
DECAY_MUTANTS = ["dg reads S_t", "A^T du misses g", "carry without decay", "prediction before decay"]


@pytest.fixture(scope="module")
def source():
    with open(oracle._SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new, count):
    assert source.count(old) == count, f"mutation '{name}' no longer matches the oracle source"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    oracle.build(str(src), so)
    lib = oracle.load(so)
    for pin in ORDER:
        try:
            ok, detail = pin(lib)
        except (FloatingPointError, ValueError, RuntimeError, ZeroDivisionError) as e:
            ok, detail = False, f"raised {e!r}"
        if not ok:
            print(f"mutant '{name}' caught by {pin.__name__}: {detail}")
            return
    pytest.fail(f"mutant '{name}' passed every pin")


def test_unmutated_copy_passes(tmp_path, source):
    """Control: the same build route with no substitution passes every pin."""
    src = tmp_path / "same.c"
    src.write_text(source)
    so = str(tmp_path / "libsame.so")
    oracle.build(str(src), so)
    lib = oracle.load(so)
    for pin in ORDER:
        ok, detail = pin(lib)
        assert ok, f"{pin.__name__}: {detail}"
    assert os.path.exists(so)


@pytest.mark.parametrize("name", DECAY_MUTANTS)
def test_strong_decay_pin_alone_catches_decay_mistakes(tmp_path, source, name):
    (old, new), = [(o, n) for m, o, n, _ in MUTANTS if m == name]
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    oracle.build(str(src), so)
    ok, detail = P.pin_strong_decay_dot_product(oracle.load(so))
    assert not ok, f"mutant '{name}' passed the strong-decay pin"
