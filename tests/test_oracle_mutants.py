"""The pins must catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of oracle/qsa_oracle.c (a dropped term, a
flipped sign, a wrong index or position, a reassociated sum, an unstable tie order ...),
builds it with the oracle's own flags, and runs the pin suite (tests/test_oracle_pins.py)
against it: at least one pin must fail.  The planted mistakes stay on the CPU; none of them
reads or writes outside the buffers the pins pass in.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qsa_oracle.c")

# (name, text in qsa_oracle.c, replacement, which occurrence (0-based)); the passage each
# mistake breaks is named in the first field
MUTANTS = [
    ("gemma gamma: (1 + w) read as w",
     "float g = 1.0f + qsa_oracle_t_to_f32(dtype, w[d]);", "float g = qsa_oracle_t_to_f32(dtype, w[d]);", 0),
    ("rms norm: eps added outside the square root",
     "float r = 1.0f / sqrtf(meanSq + eps);", "float r = 1.0f / (sqrtf(meanSq) + eps);", 0),
    ("rms norm: mean over 64 dims",
     "float meanSq = sumsq / 128.0f;", "float meanSq = sumsq / 64.0f;", 0),
    ("rope: first half rotates with +sin",
     "o[i] = a - b;", "o[i] = a + b;", 0),
    ("rope: second half rotates with -sin",
     "o[i + QSA_ROPE_HALF] = e + f;", "o[i + QSA_ROPE_HALF] = e - f;", 0),
    ("rope: sin read from the cos half",
     "float s = cs[QSA_ROPE_HALF + i];", "float s = cs[i];", 0),
    ("rope: pairs (i, i+31)",
     "#define QSA_ROPE_HALF 32 ", "#define QSA_ROPE_HALF 31 ", 0),
    ("block mean: ((k0+k1)+(k2+k3))",
     "s = s + qsa_oracle_t_to_f32(dtype, k2[d]);\n    s = s + qsa_oracle_t_to_f32(dtype, k3[d]);",
     "s = s + (qsa_oracle_t_to_f32(dtype, k2[d]) + qsa_oracle_t_to_f32(dtype, k3[d]));", 0),
    ("block mean: rows of a block read in reverse order",
     "((int64_t)QSA_COMPRESS_RATIO * g + j - pastLen)",
     "((int64_t)QSA_COMPRESS_RATIO * g + (QSA_COMPRESS_RATIO - 1 - j) - pastLen)", 0),
    ("K compress: rope at 4g + 3",
     "cosSin + (int64_t)QSA_COMPRESS_RATIO * g * 64, out);",
     "cosSin + ((int64_t)QSA_COMPRESS_RATIO * g + 3) * 64, out);", 0),
    ("block validity: an incomplete last block counted",
     "return last < ctx && first >= pastLen", "return first < ctx && first >= pastLen", 0),
    ("scores: relu dropped",
     "float rel = fmaxf(0.0f, dot);", "float rel = dot;", 0),
    ("scores: causal mask one token late",
     "int32_t nVis = (t + 1) / QSA_COMPRESS_RATIO;", "int32_t nVis = (t + 2) / QSA_COMPRESS_RATIO;", 0),
    ("scores: scaled by 1/128",
     "const float scale = 1.0f / sqrtf(128.0f);", "const float scale = 1.0f / 128.0f;", 0),
    ("scores: q heads read transposed",
     "qf[h][d] = qsa_oracle_t_to_f32(dtype, q[h * QSA_HEAD_DIM + d]);",
     "qf[h][d] = qsa_oracle_t_to_f32(dtype, q[d * QSA_NUM_Q_HEADS + h]);", 0),
    ("bf16 cast truncates",
     "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;", "(void)lower;", 0),
    ("fp16 cast rounds ties away",
     "if (rem > half || (rem == half && (kept & 1u))) kept += 1u;", "if (rem >= half) kept += 1u;", 0),
    ("selection: negative keys not inverted",
     "return (b & 0x80000000u) ? ~b : (b | 0x80000000u);",
     "return (b & 0x80000000u) ? (b & 0x7fffffffu) : (b | 0x80000000u);", 0),
    ("selection: equal keys jump ahead (unstable order)",
     "if (key[b] > key[a])", "if (key[b] >= key[a])", 0),
    ("expand: causal tail placed after 4*kSel",
     "out[QSA_COMPRESS_RATIO * kSel + j] = QSA_COMPRESS_RATIO * nVis + j;",
     "out[QSA_COMPRESS_RATIO * kSel + j] = QSA_COMPRESS_RATIO * kSel + j;", 0),
    ("pool: page row taken modulo 127",
     "int64_t row = token % QSA_PAGE_TOKENS;", "int64_t row = token % (QSA_PAGE_TOKENS - 1);", 0),
    ("decode compress: K-tails of 4g+1..4g+3",
     "k[j] = pool_tail(ps, b, 0, QSA_COMPRESS_RATIO * g + j);",
     "k[j] = pool_tail(ps, b, 0, QSA_COMPRESS_RATIO * g + j + 1);", 0),
    ("decode scores: unusable slot scores 0",
     "if (!k) { *out = -FLT_MAX; continue; }", "if (!k) { *out = 0.0f; continue; }", 0),
    ("q prep: the first padding row computed",
     "if (t >= contextLengths[b]) {", "if (t > contextLengths[b]) {", 0),
    ("q prep: rope at position t - 1",
     "cosSin + (int64_t)t * 64,", "cosSin + (int64_t)(t > 0 ? t - 1 : 0) * 64,", 0),
    ("block validity: a block starting at pastLen counted as cached",
     "return last < ctx && first >= pastLen", "return last < ctx && first > pastLen", 0),
    ("scores: the first padded row scored",
     "if (ctx <= 0 || t >= ctx) {", "if (ctx <= 0 || t > ctx) {", 0),
    ("scores: relu after the head sum",
     "float rel = fmaxf(0.0f, dot);\n      sum = sum + rel;\n    }\n    out[g] = scale * sum;",
     "float rel = dot;\n      sum = sum + rel;\n    }\n    out[g] = scale * fmaxf(0.0f, sum);", 0),
    ("scores: block g scored against kbar row g + 1",
     "const uint16_t* k = kb + (int64_t)g * QSA_HEAD_DIM;",
     "const uint16_t* k = kb + (int64_t)(g + 1 < nVis ? g + 1 : g) * QSA_HEAD_DIM;", 0),
    ("pre-decode: q rotated one position early",
     "qsa_oracle_norm_rope(dtype, x, wQ, eps, cosSin + (int64_t)pos * 64, q + h * QSA_HEAD_DIM);",
     "qsa_oracle_norm_rope(dtype, x, wQ, eps, cosSin + (int64_t)(pos > 0 ? pos - 1 : 0) * 64, q + h * QSA_HEAD_DIM);",
     0),
    ("pre-decode: the new row's raw K written to the K-tail of the previous token",
     "uint16_t* dst = pool_tail(ps, b, 0, pos);", "uint16_t* dst = pool_tail(ps, b, 0, pos - 1);", 0),
    ("pre-decode: the new row averaged first",
     "qsa_oracle_block_mean(dtype, k[0], k[1], k[2], k[3], m);",
     "qsa_oracle_block_mean(dtype, k[3], k[0], k[1], k[2], m);", 0),
    ("raw K-tail write: the last token of the incomplete block skipped",
     "t < c && t < S; ++t) {", "t < c - 1 && t < S; ++t) {", 0),
    ("decode top-k: causal tail shifted one token",
     "for (int32_t j = 0; j < tail; ++j) out[n++] = QSA_COMPRESS_RATIO * nVis + j;",
     "for (int32_t j = 0; j < tail; ++j) out[n++] = QSA_COMPRESS_RATIO * nVis + j + 1;", 0),
    ("decode top-k: split counters left as they were",
     "splitCounters[(int64_t)b * numKVHeads + h] = 0;",
     "splitCounters[(int64_t)b * numKVHeads + h] = splitCounters[(int64_t)b * numKVHeads + h];", 0),
    ("decode scores: an incomplete block counted as visible",
     "int32_t nVis = c > 0 ? c / QSA_COMPRESS_RATIO : 0;",
     "int32_t nVis = c > 0 ? (c + 3) / QSA_COMPRESS_RATIO : 0;", 0),
    ("expand: 511 blocks kept when 512 or more are visible",
     "int32_t kSel = nVis < QSA_TOPK_BLOCKS ? nVis : QSA_TOPK_BLOCKS;",
     "int32_t kSel = nVis < QSA_TOPK_BLOCKS ? nVis : QSA_TOPK_BLOCKS - 1;", 0),
]


def _mutate(text: str, old: str, new: str, occurrence: int) -> str:
    at = -1
    for _ in range(occurrence + 1):
        at = text.find(old, at + 1)
        assert at >= 0, f"mutation site not found: {old!r}"
    return text[:at] + new + text[at + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, occ, tmp_path):
    src = _mutate(open(SRC).read(), old, new, occ)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(src)
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(c_path), "-o", str(lib), "-lm"], check=True,
                   capture_output=True)
    env = dict(os.environ, QSA_ORACLE_LIBRARY=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"no pin caught '{name}':\n{r.stdout[-2000:]}"


def test_unaltered_copy_passes_every_pin(tmp_path):
    """The same harness on an unaltered copy: every pin passes (the harness itself is sound)."""
    lib = tmp_path / "libcopy.so"
    subprocess.run(["gcc", *oracle.CFLAGS, SRC, "-o", str(lib), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, QSA_ORACLE_LIBRARY=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
