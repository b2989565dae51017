"""CPU check (no GPU): the quantisers' reciprocal-and-correction division
equals IEEE binary32 division on every (amax, x) pair of BF16 values it is
used for (see quotient_proof.c).  Exhaustive: ~5.2e8 pairs, ~15 s."""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def _has_fma():
    try:
        return " fma " in open("/proc/cpuinfo").read()
    except OSError:
        return False


def test_markstein_quotient_equals_ieee_division_exhaustively():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "qproof")
        flags = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off"]
        if _has_fma():
            flags.append("-mfma")
        subprocess.run(["gcc", *flags, "-o", exe, os.path.join(HERE, "quotient_proof.c"), "-lm"],
                       check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches=0 " in r.stdout
    assert "sign_violations=0 " in r.stdout       # the sign may be applied to the E4M3 code
    pairs = int(r.stdout.split("pairs=")[1].split()[0])
    assert pairs > 5e8
