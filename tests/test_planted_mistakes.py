"""Planted-mistake check of the oracle's pins and of the parity acceptance
rules.

Each entry plants one plausible mistake in a temporary copy of ``oracle/``
or of ``tests/tolerance.py`` and runs the CPU pins (``tests/test_oracle_*.py``
and ``tests/test_tolerance_rules.py``) against it; every mistake must make
them fail.  Entries marked equivalent change nothing observable (e.g. a clamp the
next step repeats) and are listed to record that they were considered.

Under pytest the mistakes run in parallel (one process each); by hand,
``python tests/test_planted_mistakes.py`` prints the table and exits 1 if any
non-equivalent mistake survives.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (file under the repository, original text, planted text, what the mistake is, equivalent)
MUTANTS = [
    ("oracle/quant.py", "amax / np.float32(6.0)", "amax / np.float32(4.0)", "wrong E2M1 maximum in the scale", False),
    ("oracle/quant.py", "gs / sf_val", "sf_val / gs", "inverted scale reciprocal", False),
    ("oracle/quant.py", "(codes[:, 0::2] | (codes[:, 1::2] << 4))", "(codes[:, 1::2] | (codes[:, 0::2] << 4))",
     "nibble order of the packing", False),
    ("oracle/quant.py", "np.where(sf == 0, np.float32(0.0), gs / sf_val)",
     "gs / np.maximum(sf_val, np.float32(1e-30))", "zero scale not special-cased", False),
    ("oracle/quant.py", "codes[:, 0::2] = packed & 0x0F\n    codes[:, 1::2] = packed >> 4",
     "codes[:, 1::2] = packed & 0x0F\n    codes[:, 0::2] = packed >> 4", "nibble order of the unpacking", False),
    ("oracle/quant.py", "scale[..., None]).reshape(rows, k)", "scale[..., None] * 1.0009765625).reshape(rows, k)",
     "dequantized scale off by 2^-10", False),
    ("oracle/quant.py", "s = (amax / np.float32(6.0)).astype(np.float32) * gs",
     "s = (amax * gs).astype(np.float32) / np.float32(6.0)", "order of the scale's fp32 steps", False),
    ("oracle/quant.py", "return np.float32(np.float32(448.0 * 6.0) / np.float32(amax))",
     "return np.float32(np.float32(448.0 * 4.0) / np.float32(amax))", "global scale constant", False),
    ("oracle/quant.py", "gs = global_scale(amax) if amax > 0 else np.float32(1.0)",
     "gs = global_scale(amax * 2) if amax > 0 else np.float32(1.0)", "per-token global scale", False),
    ("oracle/quant.py", "row_scale[r] = np.float32(np.float32(1.0) / gs)", "row_scale[r] = gs",
     "per-token row factor not inverted", False),
    ("oracle/formats.py", "(d_hi == d_lo) & (hi % 2 == 0)", "(d_hi == d_lo) & (hi % 2 == 1)", "ties to odd", False),
    ("oracle/formats.py", "pick_hi = (d_hi < d_lo)", "pick_hi = (d_hi <= d_lo)", "ties always away from zero", False),
    ("oracle/formats.py", "mag = np.minimum(np.asarray(mag, dtype=np.float64), table[-1])",
     "mag = np.asarray(mag, dtype=np.float64)", "saturating clamp removed (the index clip repeats it)", True),
    ("oracle/formats.py", "vals.append(m / 8.0 * 2.0 ** -6)", "vals.append(m / 8.0 * 2.0 ** -7)",
     "E4M3 subnormal exponent", False),
    ("oracle/formats.py", "vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))", "vals.append((1.0 + m / 8.0) * 2.0 ** (e - 8))",
     "E4M3 exponent bias", False),
    ("oracle/formats.py", "E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)",
     "E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0)", "E2M1 value table", False),
    ("oracle/formats.py", "(np.signbit(v).astype(np.uint8) << 3)", "((v < 0).astype(np.uint8) << 3)",
     "sign of negative zero dropped", False),
    ("oracle/formats.py", "q = np.maximum(e.astype(np.int64) - 8, -133)", "q = np.maximum(e.astype(np.int64) - 9, -133)",
     "bf16 precision", False),
    ("oracle/layouts.py", ".transpose(2, 1, 0, 4, 3)[..., None]", ".transpose(2, 1, 0, 3, 4)[..., None]",
     "swizzle: scale-column dims swapped", False),
    ("oracle/layouts.py", "pad.reshape(mb, 4, 32, kb, 4)", "pad.reshape(mb, 32, 4, kb, 4)", "swizzle: row split", False),
    ("oracle/layouts.py", "dense.transpose(0, 3, 2, 1, 4)", "dense.transpose(0, 2, 3, 1, 4)", "unswizzle order", False),
    ("oracle/layouts.py", "cat = np.concatenate([up, gate], axis=0)", "cat = np.concatenate([gate, up], axis=0)",
     "gate/up interleave order", False),
    ("oracle/layouts.py", "rp, cp = _ceil(rows, 128), _ceil(c, 4)\n    pad = np.zeros",
     "rp, cp = _ceil(rows, 128), _ceil(c, 8)\n    pad = np.zeros", "scale-column padding", False),
    ("oracle/mlp.py", "d = float(np.float32(alpha)) * (a @ b.T)", "d = float(alpha) * (a @ b.T) * 1.0000001",
     "W4A4 alpha perturbed", False),
    ("oracle/mlp.py", "return (silu(gate_up[:, :i]) * gate_up[:, i:]).astype(np.float32)",
     "return (silu(gate_up[:, i:]) * gate_up[:, :i]).astype(np.float32)", "gate and up halves swapped", False),
    ("oracle/mlp.py", "return g / (1.0 + np.exp(-g))", "return g / (1.0 + np.exp(g))", "silu sign", False),
    ("oracle/mlp.py", "d = gemm_w4a4(a_packed, a_sf, w_packed, w_sf, alpha, round_bf16=False)",
     "d = gemm_w4a4(a_packed, a_sf, w_packed, w_sf, alpha, round_bf16=True)",
     "fused path rounds gate_up to bf16", False),
    ("oracle/mlp.py", "return bf16_round(silu(gate_up[:, :i]) * gate_up[:, i:])",
     "return bf16_round(np.float32(silu(gate_up[:, :i]) * gate_up[:, i:]))",
     "silu_mul_bf16 rounds through fp32", False),
    ("oracle/mlp.py", "valid = int(min(max(int(masked_m[e]), 0), g.shape[0]))",
     "valid = int(min(max(int(masked_m[e]) - 1, 0), g.shape[0]))", "masked rows off by one", False),
    ("oracle/mlp.py", "out.append(silu_mul_quant(g[:valid], gs_h))", "out.append(silu_mul_quant(g, gs_h))",
     "mask ignored", False),
    ("oracle/mlp.py", "return bf16_round(x * s)", "return bf16_round(x) * bf16_round(s)", "AWQ product not rounded", False),
    ("oracle/mlp.py", "return bf16_round(x * s)", "return bf16_round((x * s).astype(np.float32))",
     "AWQ product through fp32 (exact: 8 x 8 significant bits)", True),
    ("oracle/mlp.py", "d = float(np.float32(alpha)) * (np.asarray(x, dtype=np.float64) @ b.T)",
     "d = float(np.float32(alpha)) * (np.asarray(x, dtype=np.float64) @ b.T) * 2", "W4A16 alpha", False),
    ("oracle/mlp.py", "rs = np.asarray(a_row_scale, dtype=np.float32).astype(np.float64)[:, None]",
     "rs = np.asarray(a_row_scale, dtype=np.float32).astype(np.float64)[None, :1]",
     "per-token factor of row 0 for every row", False),
    ("tests/tolerance.py", "REL_WINDOW = 1e-3", "REL_WINDOW = 1e-1", "boundary window 100x too wide", False),
    ("tests/tolerance.py", "MAX_FLIP_FRAC = 0.005", "MAX_FLIP_FRAC = 0.5", "flip allowance 100x too large", False),
    ("tests/tolerance.py", "bad = ~((step == 1) & nb & sign_ok)", "bad = ~((step <= 2) & nb & sign_ok)",
     "two-step code flips allowed", False),
    ("tests/tolerance.py", "bad = ~((step == 1) & nb & sign_ok)", "bad = ~((step == 1) & nb)",
     "sign of a flip out of zero not checked", False),
    ("tests/tolerance.py", "assert err <= tol,", "assert err <= 10 * tol,", "GEMM bound 10x too loose", False),
    ("tests/tolerance.py", "ref_sf[sf_diff].astype(int)) == 1)", "ref_sf[sf_diff].astype(int)) <= 2)",
     "scale bytes two steps off allowed", False),
    ("tests/tolerance.py", "<= window * boundaries, axis=-1)", "<= window * 100, axis=-1)",
     "absolute instead of relative window", False),
    ("tests/tolerance.py", "diff = vg != vr ", "diff = np.abs(vg) != np.abs(vr) ", "sign flips ignored", False),
    ("tests/tolerance.py", 'assert np.all(np.isfinite(got)), f"{what}: non-finite output"', "pass",
     "explicit non-finite check removed (the bound rejects NaN and inf too)", True),
]


def run_one(fname, old, new):
    tmp = tempfile.mkdtemp()
    try:
        for d in ("oracle", "synth", "tests"):
            shutil.copytree(os.path.join(ROOT, d), os.path.join(tmp, d),
                            ignore=shutil.ignore_patterns("__pycache__"))
        path = os.path.join(tmp, fname)
        with open(path) as f:
            src = f.read()
        if src.count(old) != 1:
            return "pattern not found"
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        tests = sorted(os.path.join("tests", t) for t in os.listdir(os.path.join(tmp, "tests"))
                       if t.startswith("test_oracle") or t == "test_tolerance_rules.py")
        env = dict(os.environ, PYTHONPATH=tmp, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *tests],
                           cwd=tmp, capture_output=True, text=True, env=env)
        return "caught" if r.returncode != 0 else "survived"
    finally:
        shutil.rmtree(tmp)


def run_all():
    """[(mutant, outcome, as expected)] for every planted mistake."""
    workers = max(1, min(16, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        outcomes = list(ex.map(lambda mu: run_one(mu[0], mu[1], mu[2]), MUTANTS))
    return [(mu, res, (res == "survived") if mu[4] else (res == "caught")) for mu, res in zip(MUTANTS, outcomes)]


def test_every_planted_mistake_is_caught():
    results = run_all()
    unexpected = [f"{mu[0]}: {mu[3]} -> {res}" for mu, res, ok in results if not ok]
    assert not unexpected, "planted mistakes not caught as expected:\n" + "\n".join(unexpected)


def main():
    results = run_all()
    for (fname, _, _, what, equivalent), res, ok in results:
        print(f"{'ok ' if ok else 'BAD'} {fname:18s} {what:55s} {res}{' (equivalent)' if equivalent else ''}")
    bad = sum(not ok for _, _, ok in results)
    print(f"{len(MUTANTS)} planted mistakes, {bad} unexpected")
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
