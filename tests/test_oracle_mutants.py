"""Planted mistakes in the oracle must fail at least one pin.

Each mutant is ``pa_oracle.c`` with one plausible slip (a dropped term, a
wrong sign or index, a transposed operand, an off-by-one), built with gcc into
a temporary library and run through every pin in a child process (so that a
mutant which reads out of bounds cannot take the test run down with it).
The prefix-cache reference model (``oracle/prefix_cache.py``) gets the same
treatment with its own list of slips.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, replacement, count of occurrences expected)
MUTANTS = [
    ("floor_blocks", "int64_t n = (tokens + block_size - 1) / block_size;",
     "int64_t n = tokens / block_size;", 1),
    ("offset_from_quotient", "*offset = pos % block_size;", "*offset = pos / block_size % block_size;", 1),
    ("logical_off_by_one", "int64_t logical = pos / block_size;",
     "int64_t logical = (pos + 1) / block_size;", 1),
    ("slot_transposed", "return phys * block_size + off;", "return off * block_size + phys;", 1),
    ("dropped_scale", "x[t] = scale * dot;", "x[t] = dot;", 1),
    ("lse_drops_max", "*lse = m + log(l);", "*lse = log(l);", 1),
    ("lse_of_weights_mean", "*lse = m + log(l);", "*lse = m + log(l / (double)n_keys);", 1),
    ("exp_sign", "x[t] = exp(x[t] - m);", "x[t] = exp(m - x[t]);", 1),
    ("unnormalised", "out[i] += (x[t] / l) * values[t * d + i];", "out[i] += x[t] * values[t * d + i];", 1),
    ("values_from_keys", "const uint16_t *vrow = pool + pool_elem(p, phys, 1, kvh, off);",
     "const uint16_t *vrow = pool + pool_elem(p, phys, 0, kvh, off);", 1),
    ("gqa_interleaved", "h / group", "h % p->num_kv_heads", 5),
    ("slab_transposed", "(h * p->block_size + off) * p->head_dim",
     "(off * p->num_kv_heads + h) * p->head_dim", 1),
    ("kv_stride_single_layer", "kv * p->kv_stride",
     "kv * p->num_kv_heads * p->block_size * p->head_dim", 1),
    ("causal_off_by_one", "(int64_t)ctx_lens[s] + j + 1;", "(int64_t)ctx_lens[s] + j;", 2),
    ("decode_short_by_one", "seq_lens[s], h / group", "seq_lens[s] - 1, h / group", 2),
    ("bf16_shift", "((uint32_t)h) << 16", "((uint32_t)h) << 15", 1),
    ("writer_off_by_one", "int64_t blk = s / b, off = s % b;", "int64_t blk = s / b, off = (s + 1) % b;", 1),
    ("copy_keys_only", "for (int64_t kv = 0; kv < 2; ++kv)", "for (int64_t kv = 0; kv < 1; ++kv)", 1),
    ("copy_reversed", "pool[pool_elem(p, dst, kv, h, off) + i] = pool[pool_elem(p, src, kv, h, off) + i];",
     "pool[pool_elem(p, src, kv, h, off) + i] = pool[pool_elem(p, dst, kv, h, off) + i];", 1),
    ("swap_host_layout", "(((hb * 2 + half) * H + h) * b + off) * d", "(((hb * H + h) * 2 + half) * b + off) * d", 1),
    ("swap_direction", "if (direction == 0)", "if (direction != 0)", 1),
    ("swap_keys_only", "for (int64_t half = 0; half < 2; ++half)", "for (int64_t half = 0; half < 1; ++half)", 1),
    ("capacity_prefix_unshared", "int64_t shared = prefix / b, paged = 0;", "int64_t shared = 0, paged = 0;", 1),
    ("capacity_waste_inverted", "out[2] = 1.0 - used / reserved_slots;", "out[2] = used / reserved_slots;", 1),
    ("capacity_reserve_used", "reserved_slots += (double)max_len;", "reserved_slots += (double)lens[i];", 1),
    ("capacity_strict_budget", "reserved + max_len * bytes_per_token <= budget",
     "reserved + max_len * bytes_per_token < budget", 1),
    ("capacity_tail_from_remainder", "tail += (double)(slots - lens[i]);", "tail += (double)(b - lens[i] % b);", 1),
    ("capacity_budget_rounded_up", "int64_t free_blocks = budget / (b * bytes_per_token);",
     "int64_t free_blocks = (budget + b * bytes_per_token - 1) / (b * bytes_per_token);", 1),
]


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, count):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == count, f"mutation site for {name} not found as expected"
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(str(mutated), str(tmp_path / f"lib{name}.so"), openmp=False)
    proc = subprocess.run([sys.executable, "-m", "tests.oracle_pins", "--library", lib],
                          cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"mutant {name} passed every pin:\n{proc.stdout}{proc.stderr}"


def test_unmutated_oracle_passes_in_child(tmp_path):
    lib = oracle.build(oracle.SOURCE, str(tmp_path / "libclean.so"), openmp=False)
    proc = subprocess.run([sys.executable, "-m", "tests.oracle_pins", "--library", lib],
                          cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stdout + proc.stderr


PREFIX_MODEL = os.path.join(ROOT, "oracle", "prefix_cache.py")

# (name, original text, replacement, count of occurrences expected) in oracle/prefix_cache.py
PREFIX_MUTANTS = [
    ("prefix_block_tokens_only", "(condition, tuple(tokens[:(i + 1) * self.b]))",
     "(condition, tuple(tokens[i * self.b:(i + 1) * self.b]))", 2),
    ("prefix_condition_ignored", "key = (condition, tuple(", "key = (0, tuple(", 2),
    ("prefix_lru_newest", "victim = min(cands", "victim = max(cands", 1),
    ("prefix_stamp_root_first", "for k in reversed(chain):", "for k in chain:", 1),
    ("prefix_extensions_kept", "for k in [k for k in self.entries if k[0] == cond and k[1][:len(prefix)] == prefix]:",
     "for k in [victim]:", 1),
    ("prefix_cache_takes_no_reference", "                self.ref[blk] += 1\n                inserted += 1",
     "                inserted += 1", 1),
]


@pytest.mark.parametrize("name,old,new,count", PREFIX_MUTANTS, ids=[m[0] for m in PREFIX_MUTANTS])
def test_prefix_model_mutant_is_caught(tmp_path, name, old, new, count):
    src = open(PREFIX_MODEL).read()
    assert src.count(old) == count, f"mutation site for {name} not found as expected"
    mutated = tmp_path / f"{name}.py"
    mutated.write_text(src.replace(old, new))
    proc = subprocess.run([sys.executable, "-m", "tests.oracle_pins", "--prefix-model", str(mutated)],
                          cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"mutant {name} passed every pin:\n{proc.stdout}{proc.stderr}"
