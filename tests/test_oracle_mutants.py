"""Mutation check of the oracle's pins.

Each entry below plants one plausible mistake in a copy of the oracle (a
dropped term, a wrong sign, index or divisor, a transposed operand, a sum
where a max belongs, a reversed tie order, a wrong slice of the units), and
runs the CPU pin tests against that copy in a child process.  A mutant
passes this test only if some pin FAILS on it: a pin set that cannot tell
the mutant from the real oracle leaves that step unpinned.  No mutant reads
or writes outside the buffers its function is given (several candidate
mistakes that would have were left out), so a child process ends in a test
failure, not a crash.

Each child runs in a scratch tree holding copies of ``oracle/`` (with the
mistake), ``workloads/`` and the pin tests, so it builds and imports only
the mutated oracle.  CPU only; the mutants run in parallel, about a minute
on 8 cores.
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_pins.py", "tests/test_meank_pins.py",
        "tests/test_recover_pins.py", "tests/test_lrfu_pins.py",
        "tests/test_confidence_pins.py"]
COPIED = ["oracle/oracle.c", "oracle/__init__.py", "oracle/build.py",
          "workloads/__init__.py", "tests/conftest.py", "tests/helpers.py",
          "tests/golden/calibrate_gamma.py", "tests/golden/slot_map_example.json",
          *PINS]

# (name, the mistake it models, text in oracle/oracle.c, replacement)
C_MUTANTS = [
    # bf16 rounding
    ("bf16_truncates", "round toward zero instead of to nearest even",
     "r = ldexp(nearbyint(ldexp(m, 8)), e - 8);",
     "r = ldexp(trunc(ldexp(m, 8)), e - 8);"),
    ("bf16_subnormal_spacing", "subnormal spacing 2^-134 instead of 2^-133",
     "r = ldexp(nearbyint(ldexp(a, 133)), -133);",
     "r = ldexp(nearbyint(ldexp(a, 134)), -134);"),
    # Mean-K
    ("meank_divisor", "mean over 31 tokens",
     "orc_f64_to_bf16(sum / ORC_BLOCK)",
     "orc_f64_to_bf16(sum / (ORC_BLOCK - 1))"),
    ("meank_block_stride", "block stride of 31 tokens",
     "kraw[(r * n_tok + b * ORC_BLOCK + t) * D + d]",
     "kraw[(r * n_tok + b * (ORC_BLOCK - 1) + t) * D + d]"),
    ("meank_double_rounding", "mean rounded to fp32 before bf16",
     "orc_f64_to_bf16(sum / ORC_BLOCK)", "orc_f64_to_bf16((float)(sum / ORC_BLOCK))"),
    # Mean-K score
    ("score_no_inv_sqrt_d", "logits not scaled by 1/sqrt(D)",
     "zr[b] = dot * inv_sqrt_d;", "zr[b] = dot;"),
    ("score_sum_over_group", "sum over the GQA group instead of max",
     "if (p > best) best = p;", "best += p;"),
    ("score_mean_divisor", "mean over the window divided by G",
     "score[b] = (float)(acc / W);", "score[b] = (float)(acc / G);"),
    ("score_lse_drops_max", "LSE without its max shift",
     "lse[g * W + w] = m + log(s);", "lse[g * W + w] = log(s);"),
    ("score_blocks_reversed", "probability of block b taken from block Nb-1-b",
     "double p = exp(z[((int64_t)g * W + w) * nb + b] - lse[g * W + w]);",
     "double p = exp(z[((int64_t)g * W + w) * nb + (nb - 1 - b)] - lse[g * W + w]);"),
    ("score_q_transposed", "query read as [W][G] instead of [G][W]",
     "const uint16_t *qr = q + ((int64_t)g * W + w) * D;",
     "const uint16_t *qr = q + ((int64_t)w * G + g) * D;"),
    # QueryMemory
    ("qmem_no_token_mean", "token sum instead of mean",
     "      mean /= T;\n", "\n"),
    ("qmem_decay_gain_swapped", "decay and gain swapped",
     "v[d] = decay * (double)M[r * D + d] + gain * mean;",
     "v[d] = gain * (double)M[r * D + d] + decay * mean;"),
    ("qmem_always_renormalised", "the renorm flag ignored",
     "    if (renorm) {\n", "    if (1) {\n"),
    ("qmem_divides_by_norm_squared", "renormalised by the squared norm",
     "for (int d = 0; d < D; d++) v[d] /= n;",
     "for (int d = 0; d < D; d++) v[d] /= n2;"),
    # rule score
    ("rule_gqa_modulo", "query head hq reads KV head hq % H",
     "      int h = hq / G;\n", "      int h = hq % H;\n"),
    ("rule_no_inv_sqrt_d", "logits not scaled by 1/sqrt(D)",
     "z[j] = dot * inv_sqrt_d;", "z[j] = dot;"),
    ("rule_unnormalised", "exp(z - max) instead of the softmax",
     "if (slot_map[j] != sentinel) acc[j] += exp(z[j] - lse);",
     "if (slot_map[j] != sentinel) acc[j] += exp(z[j] - zmax);"),
    ("rule_dead_positions_scored", "dead positions not marked -1",
     "rule[j] = slot_map[j] == sentinel ? -1.0f : (float)acc[j];",
     "rule[j] = (float)acc[j];"),
    # select
    ("select_ties_high_index", "equal scores keep the higher index",
     "return (x->idx > y->idx) - (x->idx < y->idx);",
     "return (x->idx < y->idx) - (x->idx > y->idx);"),
    ("select_recent_not_forced", "recent items not in the forced set",
     "if (i < n_sink || i >= n - n_recent) {", "if (i < n_sink) {"),
    ("select_recent_off_by_one", "one recent item too few",
     "if (i < n_sink || i >= n - n_recent) {",
     "if (i < n_sink || i > n - n_recent) {"),
    ("select_mask_bit_order", "keep-mask bits in reversed order",
     "if (keep[i]) mask[i / 32] |= 1u << (i % 32);",
     "if (keep[i]) mask[i / 32] |= 1u << (31 - i % 32);"),
    # RoPE and pack
    ("rope_sign", "rotation by -angle in the first half",
     "out[j] = x[j] * c - x[j + half] * s;",
     "out[j] = x[j] * c + x[j + half] * s;"),
    ("rope_frequency", "frequency theta^(-j/D)",
     "double freq = pow(theta, -2.0 * (double)j / (double)D);",
     "double freq = pow(theta, -(double)j / (double)D);"),
    ("rope_adjacent_pairs", "element j paired with j + 1 (interleaved)",
     "    out[j] = x[j] * c - x[j + half] * s;\n"
     "    out[j + half] = x[j + half] * c + x[j] * s;\n",
     "    if (j % 2 == 0 && j + 1 < D) {\n"
     "      out[j] = x[j] * c - x[j + 1] * s;\n"
     "      out[j + 1] = x[j + 1] * c + x[j] * s;\n"
     "    }\n"
     "    out[j + half] = x[j + half];\n"),
    ("pack_tail_not_zeroed", "view tokens past the kept blocks left unwritten",
     "      for (int d = 0; d < D; d++) ko[d] = vo[d] = 0;\n", "\n"),
    ("pack_old_position", "K re-RoPEd at its old position",
     "orc_rope_f64(x, y, D, (double)(pos0 + i), theta);",
     "orc_rope_f64(x, y, D, (double)(pos0 + src), theta);"),
    ("pack_block_start_only", "every token of a block read from its first",
     "int64_t src = (int64_t)ORC_BLOCK * kept[i / ORC_BLOCK] + i % ORC_BLOCK;",
     "int64_t src = (int64_t)ORC_BLOCK * kept[i / ORC_BLOCK];"),
    # paged addressing, redirect and free
    ("slot_map_no_block_size", "physical block not multiplied by BS",
     "slot_map[p] = block_table[p / BS] * BS + p % BS;",
     "slot_map[p] = block_table[p / BS] + p % BS;"),
    ("free_ignores_prefix", "prefix slots freed",
     "if (refcnt[u] == 0 && j >= prefix_len) {", "if (refcnt[u] == 0) {"),
    ("free_ignores_aliases", "slot freed while another reference holds it",
     "if (refcnt[u] == 0 && j >= prefix_len) {", "if (j >= prefix_len) {"),
    ("redirect_sentinel_counted", "an entry already at the dead slot dropped again",
     "      if (u == sentinel) continue;\n", "\n"),
    ("redirect_skipped", "dropped positions keep their slot",
     "      *e = sentinel;\n", "\n"),
    # attention LSE and recovery score
    ("attn_lse_drops_max", "LSE without its max shift",
     "lse[l * Hq + hq] = mx + log(sum);", "lse[l * Hq + hq] = log(sum);"),
    ("attn_lse_gqa_modulo", "query head hq reads KV head hq % H",
     "      const int h = hq / G;\n", "      const int h = hq % H;\n"),
    ("attn_lse_no_inv_sqrt_d", "logits not scaled by 1/sqrt(D)",
     "s[p] = dot * inv_sqrt_d;", "s[p] = dot;"),
    ("recover_sum_over_group", "sum over the GQA group instead of max",
     "if (prob > best) best = prob;", "best += prob;"),
    ("recover_gqa_interleaved", "KV head h's group taken as heads h, h + H, ...",
     "const int hq = h * G + g;", "const int hq = g * H + h;"),
    ("recover_running_sum", "running sum instead of running mean",
     "state[p] = count == 1 ? x : state[p] + (x - state[p]) / count;",
     "state[p] = count == 1 ? x : state[p] + x;"),
    ("recover_no_lse", "probability not normalised by the LSE",
     "const double prob = exp(dot * inv_sqrt_d - lse[l * Hq + hq]);",
     "const double prob = exp(dot * inv_sqrt_d);"),
    ("recover_sees_past_seq_len", "the key at seq_len counted",
     "if (p < seq_len) {", "if (p <= seq_len && p < n_blocks * BS) {"),
    # tail compaction plan
    ("tail_region_floor", "region of floor(m/BS) blocks",
     "const int x = (m + BS - 1) / BS;", "const int x = m / BS;"),
    ("tail_dst_kept_slots", "destinations on retained slots",
     "if (!kept) dst[nd++] = p;", "if (kept) dst[nd++] = p;"),
    ("tail_freed_logical", "logical block numbers freed",
     "for (int b = 0; b < Y - x; b++) freed[b] = block_table[b];",
     "for (int b = 0; b < Y - x; b++) freed[b] = b;"),
    ("tail_mask_absolute_bit", "tail mask bit taken from the absolute position",
     "tail_mask[(p - start) / 32] |= 1u << ((p - start) % 32);",
     "tail_mask[(p - start) / 32] |= 1u << (p % 32);"),
    # LRFU keep score
    ("lrfu_no_hit_gate", "every entry gains its score",
     "ks[i] = (float)(lambda * (double)ks[i] + (hits[i] ? s : 0.0));",
     "ks[i] = (float)(lambda * (double)ks[i] + s);"),
    ("lrfu_decay_complement", "decay by 1 - lambda",
     "ks[i] = (float)(lambda * (double)ks[i] + (hits[i] ? s : 0.0));",
     "ks[i] = (float)((1.0 - lambda) * (double)ks[i] + (hits[i] ? s : 0.0));"),
    ("lrfu_negative_mass", "negative scores carry their magnitude as mass",
     "it[i].m = (s > 0.0 && isfinite(s)) ? s : 0.0;",
     "it[i].m = isfinite(s) ? fabs(s) : 0.0;"),
    ("lrfu_one_hit_too_many", "top-p prefix one entry past the mass",
     "for (int k = 0; k < n && cum < target && it[k].m > 0.0; k++) {",
     "for (int k = 0; k < n && cum <= target && it[k].m > 0.0; k++) {"),
    ("lrfu_ties_high_index", "equal scores ordered by the higher index",
     "return (x->i > y->i) - (x->i < y->i);",
     "return (x->i < y->i) - (x->i > y->i);"),
    # confidence monitor
    ("conf_divides_by_vocab", "mean over the vocabulary instead of k",
     "*conf = -top / (double)k;", "*conf = -top / (double)V;"),
    ("conf_logits_not_logprobs", "logits used as log-probabilities",
     "for (int j = 0; j < k; j++) top += sorted[j] - lse; /* log P(j) */",
     "for (int j = 0; j < k; j++) top += sorted[j];"),
    ("conf_lse_unshifted", "LSE sum not shifted by the max",
     "for (int v = 0; v < V; v++) sum += exp((double)logits[v] - mx);",
     "for (int v = 0; v < V; v++) sum += exp((double)logits[v]);"),
    ("conf_bottom_k", "the k least probable tokens",
     "qsort(sorted, (size_t)V, sizeof(double), orc_f64_desc);",
     "qsort(sorted, (size_t)V, sizeof(double), orc_f64_asc);"),
    ("trend_unit_stride", "windows at stride 1",
     "for (int i = m * s; i < m * s + w; i++)",
     "for (int i = m; i < m + w; i++)"),
    ("trend_window_last", "window's last value instead of its minimum",
     "if (conf[i] < mn) mn = conf[i];", "mn = conf[i];"),
    ("trend_keeps_upper", "entries above the percentile kept",
     "if (rp[m] <= q) {", "if (rp[m] >= q) {"),
    ("trend_percentile_ceil", "percentile rank rounded up",
     "const int lo = (int)floor(pos);", "const int lo = (int)ceil(pos);"),
    ("trend_slope_sign", "slope of the wrong sign",
     "*slope = (cnt >= 2 && den > 0.0) ? (cnt * sxy - sx * sy) / den : 0.0;",
     "*slope = (cnt >= 2 && den > 0.0) ? (sx * sy - cnt * sxy) / den : 0.0;"),
    ("budget_raised_on_rise", "budget raised on a rising trend",
     "  if (slope < 0.0) {\n", "  if (slope > 0.0) {\n"),
    ("budget_lowered_to_cap", "a budget above the cap lowered to it",
     "return nb < max_budget ? nb : (budget > max_budget ? budget : max_budget);",
     "return nb < max_budget ? nb : max_budget;"),
    ("budget_uncapped", "budget not capped",
     "return nb < max_budget ? nb : (budget > max_budget ? budget : max_budget);",
     "return nb;"),
]


# (name, the mistake it models, text in oracle/__init__.py, replacement):
# the wrappers that slice a whole event into the C functions' units
PY_MUTANTS = [
    ("score_meank_interleaved_group", "query heads h, h + H, ... grouped with KV head h",
     "score_unit(q[l, r, h * G:(h + 1) * G],", "score_unit(q[l, r, h::H],"),
    ("score_meank_layer0", "every layer scored against layer 0's Mean-K",
     "meank_all[l, h, b0:b1])", "meank_all[0, h, b0:b1])"),
    ("score_meank_softmax_from_zero", "softmax over every block before the session's end",
     "meank_all[l, h, b0:b1])", "meank_all[l, h, 0:b1])[b0:]"),
    ("select_segments_off_by_one", "each segment takes the next segment's first item",
     "a, b = int(seg_off[s]), int(seg_off[s + 1])",
     "a, b = int(seg_off[s]), int(seg_off[s + 1]) + 1"),
    ("meank_first_dim_only", "only the first leading dimension's rows averaged",
     "    rows = int(np.prod(lead)) if lead else 1\n    out = np.empty((*lead, n_tok // BLOCK",
     "    rows = lead[0] if lead else 1\n    out = np.zeros((*lead, n_tok // BLOCK"),
    ("qmem_first_dim_only", "only the first leading dimension's memories updated",
     "    rows = int(np.prod(lead)) if lead else 1\n    _check(lib().orc_qmem_update",
     "    rows = lead[0] if lead else 1\n    _check(lib().orc_qmem_update"),
]

MUTANTS = ([(n, d, "oracle/oracle.c", o, w) for n, d, o, w in C_MUTANTS] +
           [(n, d, "oracle/__init__.py", o, w) for n, d, o, w in PY_MUTANTS])


def test_every_mutation_site_is_in_the_oracle():
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))
    for name, _, path, old, new in MUTANTS:
        with open(os.path.join(ROOT, path)) as f:
            assert f.read().count(old) == 1, name
        assert old != new, name


def _run_mutant(entry, workdir):
    """Pin-test exit code of the oracle with one mistake planted (none for the
    control entry, whose path is None), and the first pin that failed."""
    name, _, path, old, new = entry
    tree = os.path.join(workdir, name)
    for rel in COPIED:
        os.makedirs(os.path.dirname(os.path.join(tree, rel)), exist_ok=True)
        shutil.copyfile(os.path.join(ROOT, rel), os.path.join(tree, rel))
    if path is not None:
        with open(os.path.join(ROOT, path)) as f:
            text = f.read().replace(old, new)
        with open(os.path.join(tree, path), "w") as f:
            f.write(text)
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    p = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-m", "not gpu",
                        "-p", "no:cacheprovider", "--rootdir", tree], cwd=tree, env=env,
                       capture_output=True, text=True, timeout=600)
    caught = re.search(r"^FAILED (\S+)", p.stdout, re.M)
    return name, p.returncode, caught.group(1) if caught else None, p.stdout[-2000:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    workers = max(1, min(8, os.cpu_count() or 1))
    control = ("control", "no mistake", None, "", "")
    with ThreadPoolExecutor(workers) as pool:
        results = list(pool.map(lambda e: _run_mutant(e, str(tmp_path)), [control, *MUTANTS]))
    _, rc, _, tail = results.pop(0)
    assert rc == 0, f"the unchanged copy fails its pins:\n{tail}"
    survivors = [(n, rc, tail) for n, rc, pin, tail in results if rc != 1 or pin is None]
    assert not survivors, "\n\n".join(f"{n}: pytest exit {rc}\n{tail}"
                                      for n, rc, tail in survivors)
