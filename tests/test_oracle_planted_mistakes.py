"""Planted mistakes: the pins are not the oracle restated.

Each case copies the oracle's C sources to a scratch folder, plants one
plausible mistake in the copy (a wrong bias, sign bit or rounding rule, a
dropped scale, a transposed layout, an off-by-one length, a broken tie rule, a
swapped operand), builds that variant and runs the oracle's pin tests against
it (``BSP_ORACLE_LIB`` points the ``oracle`` module at the variant).  At
least one pin must fail for every case.  The oracle itself is never modified;
the planted copies live only for the test.

Only mistakes in rules that the pages or the mathematics fix are planted.
Readings that no page fixes (for instance the order of the K and V fields of
several KV heads in an MXFP4 block) are consistency-checked against the GPU
path, not pinned, and are not planted here.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
sys.path.insert(0, ROOT)
from oracle import build as oracle_build  # noqa: E402

PIN_TESTS = ["tests/test_oracle_codecs.py", "tests/test_oracle_write_layout.py",
             "tests/test_oracle_pipeline.py", "tests/test_oracle_block_select.py"]

# name: (file, text in the oracle, planted text)
MISTAKES = {
    # codecs
    "e4m3 exponent bias 8": ("codecs.c", "v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                             "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3 ties away from zero": ("codecs.c", "double q = nearbyint(a / quantum);", "double q = round(a / quantum);"),
    "e4m3 not saturating": ("codecs.c", "if (v > 448.0) v = 448.0; /* satfinite */", "/* no saturation */"),
    "e2m1 sign in bit 2": ("codecs.c", "return (nib & 8) ? -v : v;", "return (nib & 4) ? -v : v;"),
    "e2m1 ties away from zero": ("codecs.c", "double v = nearbyint(a / quantum) * quantum;",
                                 "double v = round(a / quantum) * quantum;"),
    "e8m0 bias 128": ("codecs.c", "ldexp(1.0, (int)b - 127)", "ldexp(1.0, (int)b - 128)"),
    "bf16 ties away from zero": ("codecs.c", "(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    "MX shared exponent off by one": ("codecs.c", "e = (ex - 1) - 2;", "e = (ex - 1) - 1;"),
    "all-zero MX group with scale 1": ("codecs.c", "    e = -127;\n", "    e = 0;\n"),
    "e4m3 subnormals a binade low": ("codecs.c", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    # layout and writer
    "K page token-major": ("layout.c", "elem = (int64_t)(d / x) * ORC_PAGE * x + (int64_t)t * x + d % x;",
                           "elem = (int64_t)t * ORC_DIM + d;"),
    "V page token-major": ("layout.c", "elem = (int64_t)(t / x) * ORC_DIM * x + (int64_t)d * x + t % x;",
                           "elem = (int64_t)t * ORC_DIM + d;"),
    # (stays inside the block: a plant that wrote past the cache would crash, not fail a pin)
    "V pages a quarter block after K": ("layout.c",
                                        "int64_t side_base = side ? (int64_t)ORC_PAGES_PER_SIDE * id_stride : 0;",
                                        "int64_t side_base = side ? (int64_t)(ORC_PAGES_PER_SIDE / 2) * id_stride : 0;"),
    "MX nibbles swapped by the writer": ("write.c", "field[t * 64 + d / 2] = (uint8_t)(lo | (hi << 4));",
                                         "field[t * 64 + d / 2] = (uint8_t)(hi | (lo << 4));"),
    "fp8 K/V scale multiplied": ("write.c", "float q = x[d] / scale;", "float q = x[d] * scale;"),
    "fp8 index scale amax/240": ("write.c", "float s = amax > 0.0f ? amax / 448.0f : 1.0f;",
                                 "float s = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    # row lengths and scores
    "decode length off by one": ("score.c", "int64_t L = (int64_t)seq_lens[s] - (q_len - 1 - j);",
                                 "int64_t L = (int64_t)seq_lens[s] - (q_len - j);"),
    "pad rows not clamped": ("score.c", "int64_t L = (int64_t)seq_lens[s] - (q_len - 1 - j);\n      if (L < 0) L = 0;",
                             "int64_t L = (int64_t)seq_lens[s] - (q_len - 1 - j);"),
    "index head of a row from its token": ("score.c", "int h = r % Hidx;", "int h = (r / Hidx) % Hidx;"),
    "score magnitude without the absolute value": ("score.c", "adot += fabs(qv[d] * kv[d]);", "adot += qv[d] * kv[d];"),
    "prefill pad rows not clamped": ("score.c", "int64_t L = (int64_t)query_abs_pos[i] + 1;\n    if (L < 0) L = 0;",
                                     "int64_t L = (int64_t)query_abs_pos[i] + 1;"),
    "prefill length without the +1": ("score.c", "int64_t L = (int64_t)query_abs_pos[i] + 1;",
                                      "int64_t L = (int64_t)query_abs_pos[i];"),
    "fp8 index key scale dropped": ("score.c", "float kd = (float)orc_e4m3_decode(field[o * 128 + d]) * s;",
                                    "float kd = (float)orc_e4m3_decode(field[o * 128 + d]);"),
    "page score of the last token, not the max": ("score.c", "if (sc > out[p]) out[p] = sc;", "out[p] = sc;"),
    "MX index scale per 64 dims": ("score.c", "orc_e8m0_decode(field[8192 + o * 4 + d / 32])",
                                   "orc_e8m0_decode(field[8192 + o * 4 + d / 64])"),
    # selection
    "ties to the higher page": ("topk.c", "return (x->page > y->page) - (x->page < y->page);",
                                "return (x->page < y->page) - (x->page > y->page);"),
    "tail page also ranked": ("topk.c", "int n_cand = force_tail ? n - 1 : n;", "int n_cand = n;"),
    "page id from the wrong block": ("topk.c",
                                     "block_table[(int64_t)row_seq[r] * bt_stride + p / ORC_PAGES_PER_SIDE];",
                                     "block_table[(int64_t)row_seq[r] * bt_stride + p / ORC_PAGE];"),
    "block score of its first page, not the max": ("topk.c", "if (sr[p] > best) best = sr[p];", "(void)best;"),
    "MX scale bytes of a token swapped": ("write.c", "field[8192 + t * 4 + g] = sb;", "field[8192 + t * 4 + (g ^ 1)] = sb;"),
    "partial tail page counted as 16 tokens": ("topk.c",
                                               "      ti[m] = p;\n      bt[m] = (int32_t)(id_rule == 0 ? block * 16 + p % ORC_PAGES_PER_SIDE\n"
                                               "                                     : block * ORC_PAGES_PER_SIDE + p % ORC_PAGES_PER_SIDE);\n"
                                               "      ctx += (p == n - 1) ? tail_len : ORC_PAGE;",
                                               "      ti[m] = p;\n      bt[m] = (int32_t)(id_rule == 0 ? block * 16 + p % ORC_PAGES_PER_SIDE\n"
                                               "                                     : block * ORC_PAGES_PER_SIDE + p % ORC_PAGES_PER_SIDE);\n"
                                               "      ctx += ORC_PAGE;"),
    # attention
    "every token read as its page's first": ("attention.c", "int t = (int)(m % ORC_PAGE);", "int t = 0;"),
    "KV head of a sparse row from its token": ("attention.c",
                                               "    int h = r % Hkv;\n    int64_t n = sparse_ctx[r] < 0 ? 0 : sparse_ctx[r];",
                                               "    int h = (r / Hkv) % Hkv;\n    int64_t n = sparse_ctx[r] < 0 ? 0 : sparse_ctx[r];"),
    "softmax scale dropped": ("attention.c", "z[m] = (double)sm_scale * dot;", "z[m] = dot;"),
    "k and v scales swapped": ("attention.c", "(side ? v_scale : k_scale)", "(side ? k_scale : v_scale)"),
    "MX V read from the K field": ("attention.c", "kv + orc_mx_field_offset(Hkv, block, side, h);",
                                   "kv + orc_mx_field_offset(Hkv, block, 0, h);"),
    "query head row without the group": ("attention.c", "int64_t hr = r * G + i;", "int64_t hr = r + i;"),
    "dense page id at stride 8": ("attention.c", ": block * 16 + p;", ": block * 8 + p;"),
    "output not normalised": ("attention.c", "o[d] = orc_bf16_encode((float)(acc[d] / denom));",
                              "o[d] = orc_bf16_encode((float)acc[d]);"),
}


def _build_variant(name, folder):
    fname, old, new = MISTAKES[name]
    d = os.path.join(folder, "v%02d" % sorted(MISTAKES).index(name))
    shutil.copytree(ORACLE, d, ignore=shutil.ignore_patterns("*.so", "*.tmp", "__pycache__", "_planted"))
    path = os.path.join(d, fname)
    src = open(path).read()
    assert src.count(old) == 1, (name, "the planted site must occur once")
    open(path, "w").write(src.replace(old, new))
    lib = os.path.join(d, "liboracle_variant.so")
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-D_DEFAULT_SOURCE",
           "-fopenmp"] + [os.path.join(d, s) for s in oracle_build.SOURCES] + ["-o", lib, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:  # no OpenMP on this host
        r = subprocess.run([c for c in cmd if c != "-fopenmp"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return lib


def _run_pins(lib):
    env = dict(os.environ, BSP_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"]
                       + PIN_TESTS, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    failed = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
    return r.returncode, failed


@pytest.fixture(scope="module")
def outcomes():
    scratch = os.path.join(ORACLE, "_planted")  # git-ignored; removed afterwards
    os.makedirs(scratch, exist_ok=True)
    folder = tempfile.mkdtemp(prefix="run_", dir=scratch)
    try:
        names = sorted(MISTAKES)
        with cf.ThreadPoolExecutor(max(2, min(8, os.cpu_count() or 2))) as ex:
            libs = dict(zip(names, ex.map(lambda n: _build_variant(n, folder), names)))
            res = dict(zip(names, ex.map(lambda n: _run_pins(libs[n]), names)))
        yield res
    finally:
        shutil.rmtree(folder, ignore_errors=True)
        try:
            os.rmdir(scratch)  # only when no other run is using it
        except OSError:
            pass


@pytest.mark.parametrize("name", sorted(MISTAKES))
def test_a_pin_fails_on_the_planted_mistake(outcomes, name):
    rc, failed = outcomes[name]
    # exit code 1: tests ran and at least one failed (not a crash or a collection error)
    assert rc == 1, f"{name}: no pin failed (pytest exit {rc})"
    print(f"{name}: {failed[:1]}")
