"""The pins are sharp: each test here builds a copy of the oracle with one
plausible mistake planted (an off-by-one, a dropped term, a wrong sign, a wrong
tie rule, a wrong constant) and checks that the pins of that part fail on it.
Everything runs on the CPU; the product library is not involved."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "csa2_oracle.c")

# (name, exact text in the oracle, planted mistake, pin files that must catch it)
MUTANTS = [
    ("visibility_off_by_one", "return (t + 1) / m;", "return t / m;",
     ["test_oracle_formats.py", "test_oracle_index.py"]),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)",
     ["test_oracle_formats.py"]),
    ("e4m3_subnormal_scale", "ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)",
     ["test_oracle_formats.py"]),
    ("bf16_round_half_up", "u += 0x7fffu + lsb;", "u += 0x8000u;",
     ["test_oracle_formats.py"]),
    ("tail_window_bound", "win_lo[row] = s - t;", "win_lo[row] = s - t + 1;",
     ["test_oracle_tail.py"]),
    ("tail_keeps_one_row_less", "t = e < window ? e : window;",
     "t = e < window ? e : window - 1;", ["test_oracle_tail.py"]),
    ("index_relu_dropped", "acc += w * (dot > 0.0 ? dot : 0.0);", "acc += w * dot;",
     ["test_oracle_index.py"]),
    ("topk_ties_by_descending_entry", "return (x->j > y->j) - (x->j < y->j);",
     "return (x->j < y->j) - (x->j > y->j);", ["test_oracle_select.py"]),
    ("latest_block_not_kept", "chosen[keep++] = nb_all - 1;",
     "chosen[keep++] = bs[max_blocks - 1].b;", ["test_oracle_select.py"]),
    ("window_one_position_wider", "int64_t lo = t - window + 1;", "int64_t lo = t - window;",
     ["test_oracle_attn.py", "test_oracle_tail.py"]),
    ("sink_sign", "if (sink) denom += exp(sk - m);", "if (sink) denom += exp(-sk - m);",
     ["test_oracle_attn.py"]),
    ("sm_scale_dropped", "logit[i] = sm_scale * dot;", "logit[i] = dot;",
     ["test_oracle_attn.py"]),
    ("replay_one_row_short", "rp = p < window ? p : window;", "rp = p < window ? p : window - 1;",
     ["test_oracle_replay.py"]),
    ("entry_range_rounding", "entry_range[2 * r] = p / ratio;",
     "entry_range[2 * r] = (p + 1) / ratio;", ["test_oracle_replay.py"]),
    ("encode_ties_to_odd", "(d == bd && (c & 1) == 0)", "(d == bd && (c & 1) == 1)",
     ["test_oracle_quant.py"]),
    ("fp8_scale_constant", "s = amax / 448.0f;", "s = amax / 256.0f;",
     ["test_oracle_quant.py"]),
    ("mxfp4_scale_exponent", "s = ldexpf(1.0f, ex - 3);", "s = ldexpf(1.0f, ex - 2);",
     ["test_oracle_quant.py"]),
    ("mxfp4_nibble_order",
     "int nib = (d & 1) ? (byte >> 4) : (byte & 15);\n  return oracle_e2m1_value(nib) * (double)scales",
     "int nib = (d & 1) ? (byte & 15) : (byte >> 4);\n  return oracle_e2m1_value(nib) * (double)scales",
     ["test_oracle_index.py"]),
    ("fp4kv_nibble_order",
     "int nib = (d & 1) ? (byte >> 4) : (byte & 15);\n  return oracle_e2m1_value(nib) * oracle_e4m3_value",
     "int nib = (d & 1) ? (byte & 15) : (byte >> 4);\n  return oracle_e2m1_value(nib) * oracle_e4m3_value",
     ["test_oracle_fp4kv.py"]),
    ("fp4kv_scale_group", "oracle_e4m3_value(sf[d / 16]);", "oracle_e4m3_value(sf[d / 32]);",
     ["test_oracle_fp4kv.py"]),
    ("tail_source_row", "src_row[row] = (int32_t)(cu_e + e - t + k);",
     "src_row[row] = (int32_t)(cu_e + e - t + k + 1);", ["test_oracle_tail.py"]),
    ("replay_source_row", "src_row[row] = k < rp ? -1 : (int32_t)(cu_e + (k - rp));",
     "src_row[row] = k < rp ? -1 : (int32_t)(cu_e + (k - rp) + 1);", ["test_oracle_replay.py"]),
    ("pool_slot_offset", "j = blk * block + s % block;", "j = blk * block + (s + 1) % block;",
     ["test_oracle_index.py"]),
    ("head_weight_dropped", "acc += w * (dot > 0.0 ? dot : 0.0);", "acc += (dot > 0.0 ? dot : 0.0);",
     ["test_oracle_index.py"]),
    ("block_tie_order_reversed", "return (x->b > y->b) - (x->b < y->b);",
     "return (x->b < y->b) - (x->b > y->b);", ["test_oracle_select.py"]),
    ("project_drops_last_channel", "for (int d = 0; d < dim_in; ++d)",
     "for (int d = 0; d < dim_in - 1; ++d)", ["test_oracle_project.py"]),
    ("project_weight_row_offset", "w_bf16[(int64_t)o * dim_in + d]",
     "w_bf16[(int64_t)((o + 1) % dim_out) * dim_in + d]", ["test_oracle_project.py"]),
    ("project_rounds_twice", "y[i * dim_out + o] = (float)acc;",
     "y[i * dim_out + o] = (float)(float)(acc + 0x1p-30);", ["test_oracle_project.py"]),
]


@pytest.mark.parametrize("name,text,planted,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, text, planted, pins, tmp_path):
    src = open(SRC).read()
    assert src.count(text) == 1, "the mutation site moved: " + text
    mutant = tmp_path / ("oracle_%s.c" % name)
    mutant.write_text(src.replace(text, planted))
    lib = tmp_path / ("liboracle_%s.so" % name)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", str(mutant), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, CSA2_ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu",
                          "-p", "no:cacheprovider"] +
                         [os.path.join(ROOT, "tests", p) for p in pins],
                         cwd=ROOT, env=env, capture_output=True, text=True)
    assert res.returncode == 1, (name, res.returncode, res.stdout[-800:])
