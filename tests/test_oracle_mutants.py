"""Planted mistakes: every plausible slip in the oracle must fail a pin.

Each case copies oracle/mxq_oracle.c, plants one mistake (a dropped term, a
flipped tie rule, a wrong index, sign or clamp, a transposed layout factor),
builds the mutant with gcc and runs the pin suite against it in a fresh
process (MXQ_ORACLE_LIB points the oracle binding at the mutant).  The test
passes only if the pin suite fails -- or the mutant aborts on one of its own
exactness self-checks."""

import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mxq_oracle.c")

MUTANTS = {
    "scale rule: >= at the 1.5 boundary": ("(m > half ? 1 : 0)", "(m >= half ? 1 : 0)"),
    "scale rule: dropped -1": ("return (E - f.bias) - 2 + (m > half ? 1 : 0);", "return (E - f.bias) - 1 + (m > half ? 1 : 0);"),
    "scale rule: lower clamp -127": ("    if (e < -126) e = -126;\n    if (e > 125) e = 125;", "    if (e < -127) e = -127;\n    if (e > 125) e = 125;"),
    "scale rule: upper clamp 126": ("    if (e > 125) e = 125;\n", "    if (e > 125) e = 126;\n"),
    "host rule: 224 instead of 448": ("while (ldexp(448.0, s) < amax) ++s;\n    while (ldexp(448.0, s - 1) >= amax) --s;",
                                      "while (ldexp(224.0, s) < amax) ++s;\n    while (ldexp(224.0, s - 1) >= amax) --s;"),
    "host rule: floor instead of ceil": ("    while (ldexp(448.0, s - 1) >= amax) --s;", "    while (ldexp(448.0, s - 1) >= amax) --s;\n    if (ldexp(448.0, s) > amax) --s;"),
    "columnwise block of 16 rows": ("int64_t r0 = 32 * i, r1 = r0 + 32 < rows ? r0 + 32 : rows;", "int64_t r0 = 32 * i, r1 = r0 + 16 < rows ? r0 + 16 : rows;"),
    "packed MXFP4: upper clamp 125": ("            if (e > 126) e = 126;\n", "            if (e > 125) e = 125;\n"),
    "packed MXFP4: high nibble first": ("(uint8_t)(c << ((i % 2) * 4))", "(uint8_t)(c << ((1 - i % 2) * 4))"),
    "E2M1 ties to odd": ("if (dc < db || (dc == db && (c % 2) == 0)) best = c;\n    }\n    return best;\n}\n\ntypedef",
                         "if (dc < db || (dc == db && (c % 2) == 1)) best = c;\n    }\n    return best;\n}\n\ntypedef"),
    "E2M1 grid point 6 -> 5": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}"),
    "projection drops the sign": ("double val = sign_of(bits, dt) ? -mag : mag;", "double val = mag;"),
    "no non-finite poisoning": ("        if (is_nonfinite(bits, dt)) b.poisoned = 1;\n", ""),
    "MXFP8 code e + 120": ("int code = b.e + 121;", "int code = b.e + 120;"),
    "MXFP8 clamp at 1": ("            if (code < 0) code = 0;\n            scales[r * nb", "            if (code < 1) code = 1;\n            scales[r * nb"),
    "blockwise T = emax - 5": ("int T = emax - 6;", "int T = emax - 5;"),
    "blockwise clamp -126": ("            if (T < -127) T = -127;", "            if (T < -126) T = -126;"),
    "blockwise counts poisoned blocks": ("                    if (b.poisoned) continue;\n", ""),
    "E4M3 ties to odd": ("if (dc < db || (dc == db && (c % 2) == 0)) best = c;\n    }\n    return (uint8_t)",
                         "if (dc < db || (dc == db && (c % 2) == 1)) best = c;\n    }\n    return (uint8_t)"),
    "E4M3 subnormal step 2^-10": ("v = E == 0 ? ldexp((double)m, -9)", "v = E == 0 ? ldexp((double)m, -10)"),
    "E5M2 bias 16": ("ldexp((double)(4 + m), E - 17)", "ldexp((double)(4 + m), E - 18)"),
    "UE8M0 bias 126": ("return ldexp(1.0, (int)c - 127);", "return ldexp(1.0, (int)c - 126);"),
    "UE8M0 255 not NaN": ("    if (c == 255) return NAN;\n", ""),
    "swizzle factors transposed": ("(r % 32) * 16 + ((r % 128) / 32) * 4", "(r % 32) * 4 + ((r % 128) / 32) * 16"),
    "swizzle tiles per row from nb, not Cp": ("((r / 128) * (Cp / 4) + j / 4) * 512", "((r / 128) * (nb / 4) + j / 4) * 512"),
    "padded stride nb": ("if (lay == OR_PADDED) return r * Cp + j;", "if (lay == OR_PADDED) return r * nb + j;"),
    "bf16 rounding ties to odd": ("(dlo == dhi && (lo % 2) == 0)", "(dlo == dhi && (lo % 2) == 1)"),
    "partial block uses K//32": ("int64_t oracle_scale_cols(int64_t K) { return (K + 31) / 32; }",
                                 "int64_t oracle_scale_cols(int64_t K) { return K / 32 > 0 ? K / 32 : 1; }"),
}


def _run_mutant(name, old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: pattern must occur exactly once"
    tag = "".join(ch if ch.isalnum() else "_" for ch in name)
    cfile = os.path.join(tmp, f"{tag}.c")
    sofile = os.path.join(tmp, f"lib{tag}.so")
    with open(cfile, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", sofile, cfile, "-lm"])
    env = dict(os.environ, MXQ_ORACLE_LIB=sofile)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            futs = [ex.submit(_run_mutant, n, o, w, tmp) for n, (o, w) in MUTANTS.items()]
            results = dict(f.result() for f in futs)
    survivors = [n for n, rc in results.items() if rc == 0]
    assert not survivors, f"planted mistakes not caught by any pin: {survivors}"
