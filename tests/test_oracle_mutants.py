"""Plant plausible mistakes in a copy of the oracle's C source and check that the
pins catch every one of them (a dropped term, a wrong sign, a transposed
operand, a missing factor).  The mutants are compiled on the CPU only."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = [
    ("drop decay", "S[a * Dk + b] *= alpha;", "S[a * Dk + b] *= 1.0;"),
    ("erase sign", "tmp[a] = beta * (v[a] - sk);", "tmp[a] = beta * (v[a] + sk);"),
    ("drop beta", "tmp[a] = beta * (v[a] - sk);", "tmp[a] = (v[a] - sk);"),
    ("transposed readout", "acc += S[a * Dk + b] * qh[b];", "acc += S[b * Dk + a] * qh[b];"),
    ("dk sign", "dkh[b] = be * s1 - al * be * s2;", "dkh[b] = be * s1 + al * be * s2;"),
    ("dg missing alpha", "dg[r] = al * (dDP - be * dkpk);", "dg[r] = (dDP - be * dkpk);"),
    ("dS decay dropped", "D[a * Dk + b] = al * (D[a * Dk + b] - be * Dk_[a] * kh[b]);",
     "D[a * Dk + b] = (D[a * Dk + b] - be * Dk_[a] * kh[b]);"),
    ("dbeta sign", "dbeta[r] = dbe;", "dbeta[r] = -dbe;"),
    ("dq transposed", "for (int a = 0; a < Dv; ++a) acc += St[a * Dk + b] * dOt[a];",
     "for (int a = 0; a < Dv; ++a) acc += St[b * Dk + a] * dOt[a];"),
    ("norm without sqrt", "n = sqrt(s + L2EPS);", "n = (s + L2EPS);"),
    ("norm jacobian", "dk[r * Dk + b] = (dkh[b] - (k[r * Dk + b] / nk) * ck2) / nk;",
     "dk[r * Dk + b] = dkh[b] / nk;"),
]


def _checks():
    """The pins, run on square small problems (so a transposed index stays in bounds)."""
    pins.test_hand_worked_golden()
    pins.test_bruteforce_products(1, 7, 4, 4)
    pins.test_l2norm_option_matches_prenormalised()
    for l2 in (False, True):
        pins.test_backward_finite_differences_all_coords(21, 6, 3, 3, l2)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mpath = tmp_path / "mut.c"
    mpath.write_text(src.replace(old, new))
    lib_path = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(lib_path), str(mpath), "-lm"])
    real = oracle._load()
    mut = ctypes.CDLL(str(lib_path))
    mut.gdn_oracle_fwd.argtypes = real.gdn_oracle_fwd.argtypes
    mut.gdn_oracle_bwd.argtypes = real.gdn_oracle_bwd.argtypes
    mut.gdn_oracle_max_threads.restype = ctypes.c_int
    oracle._lib = mut
    try:
        with pytest.raises(AssertionError):
            _checks()
    finally:
        oracle._lib = real


def test_unmutated_passes_checks():
    _checks()
