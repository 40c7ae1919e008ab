"""Planted mistakes: every pin set must catch a plausible error in the oracle.

Each entry below is one textual mutation of ``oracle/mxoracle.c`` (a dropped
term, a wrong sign, index, constant or tie rule).  The mutated copy is built
into a temporary library and the other oracle pin tests are run against it
through ``MXORACLE_LIB``; at least one pin must fail.  Nothing here touches a
GPU or the CUDA library.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mxoracle.c")

MUTATIONS = {
 'exp_offset': ('e = (ex - 1) - 8;', 'e = (ex - 1) - 7;'),
 'tie_odd': ('(c & 1) == 0 && (best & 1) == 1', '(c & 1) == 1 && (best & 1) == 0'),
 'e2m1_sub': ('0.5 * m : ldexp(1.0 + m / 2.0, e - 1)', '1.0 * m : ldexp(1.0 + m / 2.0, e - 1)'),
 'drop_div6': ('float t = amax_b / 6.0f;', 'float t = amax_b;'),
 'bfly_sign': ('v[j + h] = a - b;', 'v[j + h] = b - a;'),
 'philox_weyl': ('W1 = 0xBB67AE85u', 'W1 = 0xBB67AE84u'),
 'nibble_order': ('if (k & 1) row[k >> 1]', 'if (!(k & 1)) row[k >> 1]'),
 'layout': ('return tile * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);', 'return tile * 512 + (r % 32) * 16 + ((r % 4)) * 4 + (c % 4);'),
 'dq_noS': ('y[r * K + k] = orc_float_to_bf16(p * S);', 'y[r * K + k] = orc_float_to_bf16(p);'),
 'sr_ge': ('code = (uint8_t)(f > u ? lo + 1 : lo);', 'code = (uint8_t)(f >= u ? lo + 1 : lo);'),
 'sr_word': ('uint32_t w = out[(i >> 1) & 3];', 'uint32_t w = out[i & 3];'),
 'recip_noclamp_zero': ('if (d == 0.0f) return 0.0f;', 'if (d == 0.0f) return FLT_MAX;'),
 'col_index': ('v[i] = bf16_to_float(x[(b * 32 + i) * ldx + c]);', 'v[i] = bf16_to_float(x[(b * 32 + i) + c * ldx]);'),
 'rht_scale': ('out[j] = v[j] * 0.25f;', 'out[j] = v[j] * 0.5f;'),
 'rht_sign_bit': ('signs[j] = ((out[0] >> j) & 1u) ? -1 : 1;', 'signs[j] = ((out[1] >> j) & 1u) ? -1 : 1;'),
 'w2d_tile_idx': ('s_tile[bo * th + bh] = bs;', 's_tile[bh * to + bo] = bs;'),
 'w2d_qcol': ('put_nibble(q_col + h * (O / 2), o, c);', 'put_nibble(q_col + o * (H / 2), h, c);'),
 'pt_amax_block': ('for (int64_t k = 0; k < H; ++k) amax = fmaxf', 'for (int64_t k = 0; k < 16; ++k) amax = fmaxf'),
 'sr_index': ('uint64_t gi = (uint64_t)(t * N_total + n_offset + n);', 'uint64_t gi = (uint64_t)(n * T + t);'),
 'sat448': ('uint8_t c = enumerate_nearest(fabs(v), orc_e4m3_value, 127, 448.0);', 'uint8_t c = enumerate_nearest(fabs(v), orc_e4m3_value, 126, 448.0);'),
 'second_scale': ('static const float NVFP4_S_DIV = 2688.0f;', 'static const float NVFP4_S_DIV = 448.0f;'),
 'fos_tie': ('int four = e4 < e6;', 'int four = e4 <= e6;'),
 'fos_div4': ('uint8_t bs4 = nvfp4_block_scale_m(amax_b, S, 4.0f);', 'uint8_t bs4 = nvfp4_block_scale_m(amax_b, S, 6.0f);'),
 'fos_sum_err': ('        err = fmaxf(err, fabsf(deq - x[i]));', '        err = err + (deq - x[i]) * (deq - x[i]);'),
 'fos_no_S': ('        float deq = prod * S;', '        float deq = prod;'),
 'bw_pow2_ge': ('while (ldexp(448.0, k) < (double)amax) ++k;', 'while (ldexp(448.0, k) <= (double)amax) ++k;'),
 'bw_div': ('float t = v[i] / sc;', 'float t = v[i] * sc;'),
 'bw_max_448': ('float sc = amax / 448.0f;', 'float sc = amax / 480.0f;'),
 'bw_zero_exp': ('if (amax == 0.0f) return -127;', 'if (amax == 0.0f) return 0;'),
 'bw_qcol': ('q_col[(rh + j) * O + ro + i] = c[i * nh + j];', 'q_col[(rh + j) * O + ro + i] = c[j * nh + i];'),
 'bw_tile_amax': ('for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(v[i]));', 'for (int i = 1; i < n; ++i) amax = fmaxf(amax, fabsf(v[i]));'),
 'dq_mx_scale': ('* orc_e8m0_value(s[r * (K / 32) + k / 32]);\n            y[r', '* orc_e8m0_value(s[r * (K / 32) + k / 32] + 1);\n            y[r'),
}


PIN_FILES = ["tests/test_oracle_formats.py", "tests/test_oracle_rng_layout.py", "tests/test_oracle_mxfp8.py",
             "tests/test_oracle_nvfp4.py", "tests/test_oracle_rht_sr.py", "tests/test_oracle_gemm_ref.py",
             "tests/test_oracle_four_over_six.py", "tests/test_oracle_blockwise_fp8.py"]


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, mutant_dir):
    src = open(SRC).read()
    before, after = MUTATIONS[name]
    assert src.count(before) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(before, after, 1)
    c_path = os.path.join(mutant_dir, name + ".c")
    so_path = os.path.join(mutant_dir, name + ".so")
    with open(c_path, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
                    c_path, "-o", so_path, "-lm"], check=True)
    env = dict(os.environ, MXORACLE_LIB=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *PIN_FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {name} survived every pin:\n{r.stdout[-2000:]}"
