"""The pins must catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of oracle.c, the kind that a
careful reading could still let through: a dropped term, a wrong sign, bias or
index, a transposed operand, a swapped nibble or layout order, a different tie
rule.  The copy is built on its own (QFP4_ORACLE_SOURCE names it), and the
CPU pin suite run against it must fail.  A control case builds the unmodified
source the same way and must pass, so a failure is due to the planted mistake
and not to the harness.  Only the CPU is used; the real oracle library is not
touched.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in oracle.c, replacement): every occurrence is replaced.
# Left out as equivalent (the result does not change): swapping the nibble
# order of A and B together in the GEMM, since elements k and k^1 always share
# a scale block and the sum pairs them the same way.
MUTANTS = [
    # rounding to the formats
    ("tie_to_odd_code", "return (lo & 1) ? hi : lo;", "return (lo & 1) ? lo : hi;"),
    ("tie_always_up", "return (lo & 1) ? hi : lo;", "return hi;"),
    ("round_toward_zero", "if (dlo < dhi) return lo;", "return lo;"),
    ("e2m1_sign_dropped", "return signbit(q) ? (mag | 8) : mag;", "return mag;"),
    # decoding
    ("e2m1_subnormal_step", "(e == 0) ? 0.5 * m :", "(e == 0) ? 1.0 * m :"),
    ("e2m1_exponent_bias", "ldexp(1.0, e - 1)", "ldexp(1.0, e - 2)"),
    ("ue8m0_exponent_bias", "ldexp(1.0, byte - 127)", "ldexp(1.0, byte - 128)"),
    ("ue4m3_exponent_bias", "(1.0 + m / 8.0) * ldexp(1.0, e - 7)", "(1.0 + m / 8.0) * ldexp(1.0, e - 8)"),
    ("ue4m3_subnormal_step", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("block_sizes_swapped", "return fmt == ORACLE_NVFP4 ? 16 : 32;", "return fmt == ORACLE_NVFP4 ? 32 : 16;"),
    ("nvfp4_b32_takes_block_16", "return fmt == ORACLE_NVFP4 ? 16 : 32;", "return fmt == ORACLE_MXFP4 ? 32 : 16;"),
    ("scale_types_swapped",
     "fmt == ORACLE_MXFP4 ? oracle_ue8m0_value(byte) : oracle_ue4m3_value(byte)",
     "fmt == ORACLE_MXFP4 ? oracle_ue4m3_value(byte) : oracle_ue8m0_value(byte)"),
    # quantiser
    ("global_scale_without_448", "return amax / 2688.0f;", "return amax / 6.0f;"),
    ("block_amax_signed",
     "if (isnan(x[i]) || isinf(x[i])) return -1;\n        float a = fabsf(x[i]);",
     "if (isnan(x[i]) || isinf(x[i])) return -1;\n        float a = x[i];"),
    ("scale_target_times_gs", "float t = (amax / 6.0f) / gs;", "float t = (amax / 6.0f) * gs;"),
    ("scale_target_without_6", "float t = (amax / 6.0f) / gs;", "float t = amax / gs;"),
    ("element_scale_without_gs", "float s = (float)oracle_scale_value(fmt, code) * gs;",
     "float s = (float)oracle_scale_value(fmt, code);"),
    ("quantise_packs_high_nibble_first", "(uint8_t)(nib[i] | (nib[i + 1] << 4))",
     "(uint8_t)((nib[i] << 4) | nib[i + 1])"),
    ("mxfp4_quantise_takes_gs", "if (fmt == ORACLE_MXFP4) gs = 1.0f;", ""),
    ("mxfp4_dequantise_takes_gs", "double gsd = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs;", "double gsd = (double)gs;"),
    ("dequantise_without_gs", "double gsd = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs;", "double gsd = 1.0;"),
    ("per_row_scale_from_first_row", "oracle_global_scale_bf16(X + m * K, K)", "oracle_global_scale_bf16(X, K)"),
    ("dequantise_high_nibble_first", "int code = (k & 1) ? (byte >> 4) : (byte & 15);",
     "int code = (k & 1) ? (byte & 15) : (byte >> 4);"),
    # scale-factor layout
    ("sf_row_split_swapped", "(rr % 32) * 16 + (rr / 32) * 4", "(rr / 32) * 16 + (rr % 32) * 4"),
    ("sf_tiles_column_major", "int64_t tile = (r / 128) * ctiles + c / 4;",
     "int64_t tile = (c / 4) * ((rows + 127) / 128) + r / 128;"),
    # GEMM
    ("gemm_b_nibble_order_only", "int cb = (k & 1) ? (bb >> 4) : (bb & 15);",
     "int cb = (k & 1) ? (bb & 15) : (bb >> 4);"),
    ("gemm_b_scale_blocks_reversed", "Bsf[n * kg + k / g]", "Bsf[n * kg + (K - 1 - k) / g]"),
    ("gemm_b_elements_reversed", "int bb = B[n * (K / 2) + k / 2];", "int bb = B[n * (K / 2) + (K - 1 - k) / 2];"),
    ("gemm_a_scale_block_of_16", "Asf[m * kg + k / g]", "Asf[m * kg + k / 16]"),
    ("gemm_drops_global_scale", "*d_out = gsab * acc;", "*d_out = acc;"),
    ("mxfp4_gemm_takes_gs", "double gsab = fmt == ORACLE_MXFP4 ? 1.0 : (double)gs_a * (double)gs_b;",
     "double gsab = (double)gs_a * (double)gs_b;"),
    ("gemm_global_scale_of_a_twice", "(double)gs_a * (double)gs_b", "(double)gs_a * (double)gs_a"),
    ("gemm_accumulates_in_fp32", "double acc = 0.0, tacc = 0.0;", "float acc = 0.0f; double tacc = 0.0;"),
    # SwiGLU and the array roundings behind the requantisation check
    ("swiglu_sigmoid_of_plus_g", "G[i] * U[i] / (1.0 + exp(-G[i]))", "G[i] * U[i] / (1.0 + exp(G[i]))"),
    ("swiglu_sigmoid_of_up", "G[i] * U[i] / (1.0 + exp(-G[i]))", "G[i] * U[i] / (1.0 + exp(-U[i]))"),
    ("swiglu_without_sigmoid", "G[i] * U[i] / (1.0 + exp(-G[i]))", "G[i] * U[i]"),
    ("swiglu_half_sigmoid", "G[i] * U[i] / (1.0 + exp(-G[i]))", "G[i] * U[i] / (2.0 + exp(-G[i]))"),
    ("e2m1_round_n_drops_sign", "code[i] = (uint8_t)oracle_e2m1_round(q[i]);",
     "code[i] = (uint8_t)(oracle_e2m1_round(q[i]) & 7);"),
    ("scale_round_n_other_format", "code[i] = (uint8_t)oracle_scale_round(fmt, t[i]);",
     "code[i] = (uint8_t)oracle_scale_round(1 - fmt, t[i]);"),
    ("scale_codes_bits_without_gs",
     "float t = (amax / 6.0f) / gs;\n        code[i] = (uint8_t)oracle_scale_round(fmt, t);",
     "float t = amax / 6.0f;\n        code[i] = (uint8_t)oracle_scale_round(fmt, t);"),
    ("element_codes_bits_multiplies", "float q = float_of_bits(first + (uint32_t)i) / s;",
     "float q = float_of_bits(first + (uint32_t)i) * s;"),
    ("element_codes_bits_off_by_one", "float q = float_of_bits(first + (uint32_t)i) / s;",
     "float q = float_of_bits(first + (uint32_t)i + 1) / s;"),
    # residual add and RMSNorm
    ("bf16_round_truncates", "return (uint16_t)((u + 0x7FFFu + lsb) >> 16);", "return (uint16_t)(u >> 16);"),
    ("bf16_round_ties_up", "return (uint16_t)((u + 0x7FFFu + lsb) >> 16);", "return (uint16_t)((u + 0x8000u) >> 16);"),
    ("rmsnorm_sum_not_mean", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / sqrt(ss + eps)"),
    ("rmsnorm_eps_outside_sqrt", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / (sqrt(ss / (double)K) + eps)"),
    ("rmsnorm_gamma_dropped", "* inv * (double)bf16_bits_to_float(gamma[k]);", "* inv;"),
    ("rmsnorm_residual_ignored", "const float s = r ? xv + bf16_bits_to_float(r[m * K + k]) : xv;",
     "const float s = xv;"),
    # 2:4 pair-granular sparse operand
    ("sparse24_even_group_high_nibble", "(meta[r * (K / 16) + j / 2] >> (4 * (j & 1))) & 15",
     "(meta[r * (K / 16) + j / 2] >> (4 - 4 * (j & 1))) & 15"),
    ("sparse24_kept_bytes_swapped",
     "w[i0] = Wc[r * (K / 4) + 2 * j];\n            w[i1] = Wc[r * (K / 4) + 2 * j + 1];",
     "w[i1] = Wc[r * (K / 4) + 2 * j];\n            w[i0] = Wc[r * (K / 4) + 2 * j + 1];"),
    ("sparse24_negative_zero_is_nonzero", "return (b & 7) == 0 && ((b >> 4) & 7) == 0;", "return b == 0;"),
    ("sparse24_group_stride_halved", "uint8_t *w = W + r * (K / 2) + 4 * j;\n            for (int i = 0; i < 4; ++i) w[i] = 0;",
     "uint8_t *w = W + r * (K / 2) + 2 * j;\n            for (int i = 0; i < 4; ++i) w[i] = 0;"),
    ("sparse24_meta_indices_swapped", "(uint8_t)((idx[0] | (idx[1] << 2)) << (4 * (j & 1)))",
     "(uint8_t)((idx[1] | (idx[0] << 2)) << (4 * (j & 1)))"),
    ("rescale_row_twice", "(cs ? (double)cs[n] : 1.0)", "(rs ? (double)rs[m] : 1.0)"),
    ("rescale_drops_column", "(cs ? (double)cs[n] : 1.0)", "1.0"),
]


# The same for the Python half of the oracle (oracle/__init__.py): the
# marshalling wrappers and the requantisation check.  Left out: rounding the
# box ends to nearest instead of outward (equivalent: an fp32 value inside
# the real box is never outside its nearest-rounded ends).
PY_MUTANTS = [
    ("py_quantize_bf16_read_as_fp32",
     "    if x.dtype == np.uint16:\n        rc = lib.oracle_quantize_bf16(",
     "    if x.dtype == np.int64:\n        rc = lib.oracle_quantize_bf16("),
    ("py_quantize_per_row_scales_ignored", "    if np.ndim(gs) == 1:\n        if x.dtype != np.uint16:",
     "    if False:\n        if x.dtype != np.uint16:"),
    ("py_swiglu_gate_and_up_swapped",
     "    G, TG = gemm_nt(fmt, A, A_sf, Wg, Wg_sf, gs_a, gs_w)\n    U, TU = gemm_nt(fmt, A, A_sf, Wu, Wu_sf, gs_a, gs_w)",
     "    G, TG = gemm_nt(fmt, A, A_sf, Wu, Wu_sf, gs_a, gs_w)\n    U, TU = gemm_nt(fmt, A, A_sf, Wg, Wg_sf, gs_a, gs_w)"),
    ("py_requant_negative_zero_equals_positive", "key[8] = -1.0", "key[8] = 0.0"),
    ("py_requant_scale_range_ignores_interval", "code_lo = _scale_round_n(fmt, (amax_lo / six) / gs_hi)",
     "code_lo = _scale_round_n(fmt, (amax_lo / six) / gs_lo)"),
    ("py_requant_element_range_ignores_interval", "corners.min(axis=0)", "corners[0]"),
    ("py_requant_box_never_spans_zero",
     "a_small = np.where((lo <= 0) & (hi >= 0), np.float32(0), np.minimum(np.abs(lo), np.abs(hi)))",
     "a_small = np.minimum(np.abs(lo), np.abs(hi))"),
    ("py_requant_zero_scale_not_special", "el_ok = np.where(zero, nib == 0,", "el_ok = np.where(False, nib == 0,"),
    ("py_rows_global_scale_without_6", "max(axis=1) / 2688.0", "max(axis=1) / 448.0"),
]

PKG = os.path.join(ROOT, "oracle")


def _run_py(workdir, init_text):
    """Run the pin suite against a copy of the oracle package whose Python
    half is init_text: the copy and a copy of the pin suite (with its
    conftest, which puts the copy first on sys.path) live in workdir."""
    os.makedirs(os.path.join(workdir, "oracle"), exist_ok=True)
    shutil.copy(os.path.join(PKG, "oracle.c"), os.path.join(workdir, "oracle", "oracle.c"))
    with open(os.path.join(workdir, "oracle", "__init__.py"), "w") as f:
        f.write(init_text)
    tdir = os.path.join(workdir, "tests")
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(tdir, "golden"), dirs_exist_ok=True)
    for name in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", name), os.path.join(tdir, name))
    env = dict(os.environ, PYTHONPATH=ROOT, OMP_NUM_THREADS="2")
    env.pop("QFP4_ORACLE_SOURCE", None)
    b = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__); oracle.build(force=True)"],
                       cwd=workdir, env=env, capture_output=True, text=True, timeout=300)
    if b.returncode != 0 or not b.stdout.strip().startswith(os.path.join(workdir, "oracle")):
        return b.returncode or -1, None, (b.stdout + b.stderr)[-2000:]
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(tdir, "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=workdir, env=env, capture_output=True, text=True,
                       timeout=300)
    return 0, r.returncode, r.stdout[-2000:]


def _run(workdir, text):
    """Build the given oracle source in workdir and run the pin suite on it.
    Returns (build returncode, pin-suite returncode, pin-suite output)."""
    os.makedirs(workdir, exist_ok=True)
    src = os.path.join(workdir, "oracle.c")
    with open(src, "w") as f:
        f.write(text)
    env = dict(os.environ, QFP4_ORACLE_SOURCE=src, OMP_NUM_THREADS="2")
    b = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.build(force=True))"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    if b.returncode != 0 or os.path.dirname(b.stdout.strip()) != workdir:
        return b.returncode or -1, None, b.stderr[-2000:]
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    return 0, r.returncode, r.stdout[-2000:]


def test_unmodified_copy_passes(tmp_path):
    with open(SRC) as f:
        brc, rc, out = _run(str(tmp_path), f.read())
    assert brc == 0, out
    assert rc == 0, out


def test_planted_mistakes_are_caught(tmp_path):
    with open(SRC) as f:
        text = f.read()
    for name, old, new in MUTANTS:
        assert old in text, f"{name}: text to mutate not found in oracle.c"
    jobs = {name: (str(tmp_path / name), text.replace(old, new)) for name, old, new in MUTANTS}
    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(workers) as pool:
        results = dict(zip(jobs, pool.map(lambda j: _run(*j), jobs.values())))
    not_built = {n: r[2] for n, r in results.items() if r[0] != 0}
    assert not not_built, f"mutants that did not build: {not_built}"
    # pytest exit code 1 = some pin failed; 0 = survived; anything else (a
    # usage error or a crash) does not count as caught
    survived = {n: r[2] for n, r in results.items() if r[1] != 1}
    assert not survived, "mistakes the pins let through:\n" + "\n".join(
        f"{n}:\n{out}" for n, out in survived.items())


def test_unmodified_python_copy_passes(tmp_path):
    with open(os.path.join(PKG, "__init__.py")) as f:
        brc, rc, out = _run_py(str(tmp_path), f.read())
    assert brc == 0, out
    assert rc == 0, out


def test_planted_python_mistakes_are_caught(tmp_path):
    with open(os.path.join(PKG, "__init__.py")) as f:
        text = f.read()
    for name, old, new in PY_MUTANTS:
        assert old in text, f"{name}: text to mutate not found in oracle/__init__.py"
    jobs = {name: (str(tmp_path / name), text.replace(old, new)) for name, old, new in PY_MUTANTS}
    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(workers) as pool:
        results = dict(zip(jobs, pool.map(lambda j: _run_py(*j), jobs.values())))
    not_built = {n: r[2] for n, r in results.items() if r[0] != 0}
    assert not not_built, f"copies that did not import or build: {not_built}"
    survived = {n: r[2] for n, r in results.items() if r[1] != 1}
    assert not survived, "mistakes the pins let through:\n" + "\n".join(
        f"{n}:\n{out}" for n, out in survived.items())
