"""The oracle's pins are sensitive: each plausible mistake planted in a copy of the oracle
(on the CPU, in a temporary file) makes the pin suite fail."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "ratio_inverted": ("return min(1.0, p / q)", "return min(1.0, q / p) if p > 0 else 0.0"),
    "accept_compare_inverted": ("return bool(u < ratio), abs(u - ratio)", "return bool(u >= ratio), abs(u - ratio)"),
    "residual_sign": ("return np.maximum(0.0, P - Q)", "return np.maximum(0.0, Q - P)"),
    "no_prefix_counts": ("    for t in prefix:\n        c[int(t)] += 1\n", ""),
    "no_renorm_topp": ("pk = w / w.sum()", "pk = w / weights.sum()"),
    "presence_sign": ("pen = (pen + p).astype(np.float32)", "pen = (pen - p).astype(np.float32)"),
    "cdf_non_strict": ("hits = np.nonzero(C > target)[0]", "hits = np.nonzero(C >= target)[0]"),
    "topk_off_by_one": ("tau_k = values[order[top_k - 1]]", "tau_k = values[order[top_k]]"),
    "draft_temperature_missing": ("w = q ** (1.0 / float(T))", "w = q"),
    "bonus_wrong_position": ("        P = dist(\"nucleus_p\", a)\n",
                             "        P = dist(\"nucleus_p\", max(a - 1, 0))\n"),
    "logprob_penalised": ("row = xp(j) if batch.logprob_mode == \"penalised\" else x[j]", "row = xp(j)"),
    "penalised_mode_ignored": ("row = xp(j) if batch.logprob_mode == \"penalised\" else x[j]", "row = x[j]"),
    "sparse_ids_ignored": ("out[np.asarray(batch.q_ids[b, i], np.int64)] = batch.q[b, i]",
                           "out[np.arange(batch.q.shape[-1])] = batch.q[b, i]"),
    "d2t_sign": ("out[dv + np.asarray(batch.d2t, np.int64)] = batch.q[b, i]",
                 "out[dv - np.asarray(batch.d2t, np.int64)] = batch.q[b, i]"),
    "layout_check_skipped": ("if T > 0 and K > 0 and not draft_layout_ok(batch, b, K):", "if False:"),
    "eos_draft_excluded": ("            a = int(hit[0]) + 1\n", "            a = int(hit[0])\n"),
    "rejected_position_not_attempted": ("attempted[:min(a + 1, K)] = 1", "attempted[:a] = 1"),
    "draw_margin_in_mass_units": ("return t, float(min(target - lo, C[t] - target) / total)",
                                  "return t, float(min(target - lo, C[t] - target))"),
    "admissible_without_slack": ("(lo < float(u) + eps) & (hi > float(u) - eps)", "(lo <= float(u)) & (hi > float(u))"),
    "accept_flip_ignored": ("                acc = not acc\n", "                acc = acc\n"),
    "nucleus_flip_ignored": ("    if flip == \"drop_last\" and nk > 1:\n        nk -= 1\n",
                             "    if flip == \"drop_last\" and nk > 1:\n        nk -= 0\n"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "epilogue.py")).read()
    a, b = MUTATIONS[name]
    assert a in src
    mut = tmp_path / "epilogue_mut.py"
    mut.write_text(src.replace(a, b, 1))
    code = textwrap.dedent(f"""
        import sys, importlib.util
        sys.path.insert(0, {ROOT!r})
        spec = importlib.util.spec_from_file_location('oracle.epilogue', {str(mut)!r})
        m = importlib.util.module_from_spec(spec)
        sys.modules['oracle.epilogue'] = m
        spec.loader.exec_module(m)
        import oracle
        oracle.epilogue = m
        import pytest
        sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider',
                              {os.path.join(ROOT, 'tests', 'test_oracle_pins.py')!r},
                              {os.path.join(ROOT, 'tests', 'test_oracle_extensions.py')!r}]))
    """)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode != 0, f"mutation {name} survived:\n{r.stdout[-2000:]}"
