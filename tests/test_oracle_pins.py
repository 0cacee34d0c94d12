"""The fp64 oracle against its pins (CPU only), and the pins against planted mistakes.

The mutation tests copy oracle/pa_oracle.c to a temporary directory, plant one
plausible mistake (a dropped term, a wrong sign, a transposed index, the
literal unnormalised partition output, ...), build it, and require that at
least one pin fails.  Every planted mistake keeps all memory accesses in bounds.
"""
import json
import pathlib
import subprocess
import sys

import pytest

import oracle
import oracle_pins as P

ROOT = pathlib.Path(__file__).resolve().parents[1]


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(lambda w, **kw: oracle.oracle_decode(w, **kw))


# (name, original text, replacement, occurrences to replace (0 = all))
MUTATIONS = [
    ("drop_scale", "double z = a->scale * dot;", "double z = dot;", 0),
    ("gqa_modulo", "const int kvh = h / group;", "const int kvh = h % a->num_kv_heads;", 0),
    ("split_key_transposed",
     "return base + ((int64_t)(d / x) * a->block_size + o) * x + (d % x);",
     "return base + ((int64_t)o * (a->head_size / x) + d / x) * x + (d % x);", 0),
    ("split_value_transposed", "return base + (int64_t)d * a->block_size + o;",
     "return base + (int64_t)o * a->head_size + d;", 0),
    ("nhd_key_transposed", "    /* NHD: [block_size][head_size] */\n    return base + (int64_t)o * a->head_size + d;",
     "    return base + (int64_t)d * a->block_size + o;", 0),
    ("alibi_sign", "z += (double)a->alibi_slopes[h] * (double)t;",
     "z -= (double)a->alibi_slopes[h] * (double)t;", 0),
    ("alibi_partition_relative", "z += (double)a->alibi_slopes[h] * (double)t;",
     "z += (double)a->alibi_slopes[h] * (double)(t % a->partition_size);", 0),
    ("softcap_clamp", "z = a->softcap * tanh(z / a->softcap);",
     "z = z < a->softcap ? z : a->softcap;", 0),
    ("softcap_no_tanh", "z = a->softcap * tanh(z / a->softcap);",
     "z = a->softcap * (z / a->softcap);", 0),
    ("tmp_unnormalised", "for (int d = 0; d < d_sz; ++d) sc->vrow[d] /= e;", "", 0),
    ("exp_sum_global_max", "double w = exp(sc->z[t] - m);", "double w = exp(sc->z[t] - M);", 0),
    ("partition_drops_last_token", "t1 = t0 + PS < len ? t0 + PS : len;",
     "t1 = t0 + PS - 1 < len ? t0 + PS - 1 : len;", 0),
    ("query_rows_transposed", "const int64_t qoff = (row * a->num_heads + h) * d_sz;",
     "const int64_t qoff = ((int64_t)h * a->num_query_tokens + row) * d_sz;", 0),
    ("slot_off_by_one", "        int o = t % a->block_size;\n        double dot",
     "        int o = (t + 1) % a->block_size;\n        double dot", 0),
    ("reduce_weight_without_exp_sum", "double r = exp(m - M) * e;", "double r = exp(m - M);", 0),
    ("half_exponent_bias", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);", 0),
    ("window_off_by_one", "t_lo = len - 1 - a->window_left;", "t_lo = len - a->window_left;", 0),
    ("window_ignored", "    if (a->window_left >= 0 && len - 1 - a->window_left > 0) t_lo = len - 1 - a->window_left;\n", "", 0),
    ("scales_swapped", "(a->k_scale * load_elem(a->key_cache", "(a->v_scale * load_elem(a->key_cache", 0),
    ("e4m3_bias", "else v = ldexp((double)(8 + f), e - 10);", "else v = ldexp((double)(8 + f), e - 11);", 0),
    ("e5m2_subnormal", "v = ldexp((double)f, -16);", "v = ldexp((double)f, -15);", 0),
    ("fp8_split_packing", "int x = 16 / elem_bytes(cache_dtype(a));", "int x = 16 / elem_bytes(a->dtype);", 0),
    ("causal_ignored", "const int len = a->seq_lens[s] - qn + 1 + qi;", "const int len = a->seq_lens[s];", 0),
    ("query_tokens_reversed", "const int len = a->seq_lens[s] - qn + 1 + qi;",
     "const int len = a->seq_lens[s] - qi;", 0),
    ("unused_partition_sum_one", "if (a->exp_sums) a->exp_sums[stat_off + p] = 0.0;",
     "if (a->exp_sums) a->exp_sums[stat_off + p] = 1.0;", 0),
]


@pytest.mark.parametrize("name,old,new,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, count):
    src = (ROOT / "oracle" / "pa_oracle.c").read_text()
    assert old in src, f"mutation target for {name} not found in pa_oracle.c"
    mutated = src.replace(old, new) if count == 0 else src.replace(old, new, count)
    (tmp_path / "pa_oracle.c").write_text(mutated)
    lib = oracle.compile_source(tmp_path / "pa_oracle.c", tmp_path / f"lib_{name}.so")
    proc = subprocess.run([sys.executable, str(ROOT / "tests" / "oracle_pins.py"), str(lib)],
                          capture_output=True, text=True, timeout=600, cwd=str(ROOT))
    assert proc.returncode in (0, 1), proc.stderr[-2000:]
    report = json.loads(proc.stdout.strip().splitlines()[-1])
    failed = [k for k, v in report.items() if v]
    assert failed, f"planted mistake {name} passed every pin"
