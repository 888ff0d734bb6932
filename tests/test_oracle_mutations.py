"""The oracle's pins catch planted mistakes (CPU only).

Each case plants one plausible mistake in a copy of the oracle -- a dropped
term, a wrong sign, base, position, index, operand or order -- builds that
copy with gcc in a temporary folder, and runs every pin of
``test_oracle_pins.py`` against it in a child process.  Every planted mistake
must fail at least one pin, and the unchanged copy must pass them all.  The
mistakes are chosen so that every memory access of the mutant stays in
bounds on the pins' inputs: a mutant fails by an assertion, never by a crash.
"""
import json
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")
ORACLE = os.path.join(ROOT, "oracle")
C, PY = "kvx_oracle.c", "__init__.py"

# name -> list of (file, original text, planted text, occurrences replaced)
MUTATIONS = {
    "unchanged": [],
    # half-split RoPE
    "rope_angle_ignores_direction": [
        (C, "double a = (double)sign * pos * w;", "double a = pos * w;", 1)],
    "rope_frequency_theta_pow_minus_i_over_d": [
        (C, "pow(theta, -2.0 * (double)i / (double)d)", "pow(theta, -1.0 * (double)i / (double)d)",
         1)],
    "rope_rotation_transposed": [
        (C, "out[i] = x0 * c - x1 * s;\n    out[i + half] = x0 * s + x1 * c;",
         "out[i] = x0 * c + x1 * s;\n    out[i + half] = -x0 * s + x1 * c;", 1)],
    "rope_interleaved_pairs": [
        (C, "double x0 = x[i], x1 = x[i + half];\n    out[i] = x0 * c - x1 * s;\n"
            "    out[i + half] = x0 * s + x1 * c;",
         "double x0 = x[2 * i], x1 = x[2 * i + 1];\n    out[2 * i] = x0 * c - x1 * s;\n"
         "    out[2 * i + 1] = x0 * s + x1 * c;", 1)],
    # per-head map of one token
    "unrotate_with_target_base": [
        (C, "kvxo_rope(src_k_rows[j], d, p_src, theta_src, -1, xk + j * d);",
         "kvxo_rope(src_k_rows[j], d, p_src, theta_tgt, -1, xk + j * d);", 1)],
    "rerotate_with_source_base": [
        (C, "kvxo_rope(yk, d, p_tgt, theta_tgt, +1, out_k);",
         "kvxo_rope(yk, d, p_tgt, theta_src, +1, out_k);", 1)],
    "rerotate_at_source_position": [
        (C, "kvxo_rope(yk, d, p_tgt, theta_tgt, +1, out_k);",
         "kvxo_rope(yk, d, p_src, theta_tgt, +1, out_k);", 1)],
    "key_not_rerotated": [
        (C, "kvxo_rope(yk, d, p_tgt, theta_tgt, +1, out_k);",
         "memcpy(out_k, yk, sizeof(double) * (size_t)d);", 1)],
    "values_unrotated_like_keys": [
        (C, "for (int c = 0; c < d; ++c) xv[j * d + c] = src_v_rows[j][c];",
         "kvxo_rope(src_v_rows[j], d, p_src, theta_src, -1, xv + j * d);", 1)],
    "value_bias_dropped": [(C, "out_v[n] = bv[n];", "out_v[n] = 0.0;", 1)],
    "key_bias_added_after_rerotation": [
        (C, "yk[n] = bk[n];", "yk[n] = 0.0;", 1),
        (C, "kvxo_rope(yk, d, p_tgt, theta_tgt, +1, out_k);",
         "kvxo_rope(yk, d, p_tgt, theta_tgt, +1, out_k);\n"
         "  for (int n = 0; n < d; ++n) out_k[n] += bk[n];", 1)],
    "value_map_uses_key_weights": [
        (C, "out_v[n] += xv[q] * wv_row[n];", "out_v[n] += xv[q] * wk_row[n];", 1)],
    "selected_layers_concatenated_in_reverse": [
        (C, "kvxo_rope(src_k_rows[j], d, p_src", "kvxo_rope(src_k_rows[k - 1 - j], d, p_src", 1),
        (C, "xv[j * d + c] = src_v_rows[j][c];", "xv[j * d + c] = src_v_rows[k - 1 - j][c];", 1)],
    # routing of the whole transfer
    "key_rows_read_from_mirrored_head": [
        (C, "krows[j] = P->src_k + ((s * src_rows + srow) * H + h) * d;",
         "krows[j] = P->src_k + ((s * src_rows + srow) * H + (H - 1 - h)) * d;", 1)],
    "key_and_value_maps_swapped": [
        (C, "const double *Wk = P->w + ((lt * H + h) * 2 + 0) * kd * d;",
         "const double *Wk = P->w + ((lt * H + h) * 2 + 1) * kd * d;", 1),
        (C, "const double *Wv = P->w + ((lt * H + h) * 2 + 1) * kd * d;",
         "const double *Wv = P->w + ((lt * H + h) * 2 + 0) * kd * d;", 1)],
    "target_offset_ignored": [
        (C, "int64_t pt = P->tgt_pos ? P->tgt_pos[g] : p + off;",
         "int64_t pt = P->tgt_pos ? P->tgt_pos[g] : p + 0 * off;", 3)],
    "source_position_counted_from_batch_start": [
        (C, "int64_t p = P->src_pos ? P->src_pos[g] : g - beg;",
         "int64_t p = P->src_pos ? P->src_pos[g] : g;", 4)],
    "backwards_request_table_accepted": [
        (C, "if (P->cu_seqlens[r + 1] < P->cu_seqlens[r]) ok = 0;",
         "if (P->cu_seqlens[r + 1] < P->cu_seqlens[r]) ok = ok + 0;", 5)],
    "contiguous_row_ignores_request_slab": [
        (C, "return r * dst_capacity + p_tgt;", "return 0 * r * dst_capacity + p_tgt;", 1)],
    "paged_target_slot_off_by_one": [
        (C, "return phys * block_size + p_tgt % block_size;",
         "return phys * block_size + (p_tgt + 1) % block_size;", 1)],
    "paged_source_slot_off_by_one": [
        (C, "return phys * block_size + p % block_size;",
         "return phys * block_size + (p + 1) % block_size;", 1)],
    # wide-feature map
    "wide_features_values_before_keys": [
        (C, "x + ((int64_t)(j * 2 + 0) * H + h) * d);", "x + ((int64_t)(j * 2 + 1) * H + h) * d);",
         1),
        (C, "x[((int64_t)(j * 2 + 1) * H + h) * d + i]", "x[((int64_t)(j * 2 + 0) * H + h) * d + i]",
         1)],
    "wide_features_head_major": [
        (C, "x + ((int64_t)(j * 2 + 0) * H + h) * d);", "x + ((int64_t)(j * H + h) * 2 + 0) * d);",
         1),
        (C, "x[((int64_t)(j * 2 + 1) * H + h) * d + i]", "x[((int64_t)(j * H + h) * 2 + 1) * d + i]",
         1)],
    "wide_outputs_kind_major": [
        (C, "y + (int64_t)(h * 2 + 0) * d, d, p_tgt", "y + (int64_t)(0 * H + h) * d, d, p_tgt", 1),
        (C, "y + (int64_t)(h * 2 + 1) * d, sizeof", "y + (int64_t)(1 * H + h) * d, sizeof", 1)],
    "wide_keys_not_unrotated": [
        (C, "kvxo_rope(src_k_rows[j] + (int64_t)h * d, d, p_src, theta_src, -1,",
         "kvxo_rope(src_k_rows[j] + (int64_t)h * d, d, 0.0 * p_src, theta_src, -1,", 1)],
    # fidelity diagnostics
    "diag_key_content_not_unrotated": [
        (C, "kvxo_rope(y, (int)d, (double)pt, P->theta_tgt, -1, content);",
         "memcpy(content, y, sizeof(double) * (size_t)d);", 1)],
    "diag_key_content_rotated_forward": [
        (C, "kvxo_rope(y, (int)d, (double)pt, P->theta_tgt, -1, content);",
         "kvxo_rope(y, (int)d, (double)pt, P->theta_tgt, +1, content);", 1)],
    "diag_cosine_normalised_by_reference_only": [
        (C, "st[1] += dot / sqrt(aa * yy);", "st[1] += dot / yy;", 1)],
    "diag_residual_as_energy_difference": [
        (C, "res += (y[i] - a[i]) * (y[i] - a[i]);", "res += y[i] * y[i] - a[i] * a[i];", 1)],
    "diag_zero_vector_cosine_one": [
        (C, "if (aa > 0.0 && yy > 0.0) st[1] += dot / sqrt(aa * yy);",
         "st[1] += (aa > 0.0 && yy > 0.0) ? dot / sqrt(aa * yy) : 1.0;", 1)],
    "explained_variance_uncentred": [
        (PY, "ss_tot = s[..., 3] - np.sum(s[..., 4:] ** 2, axis=-1) / n",
         "ss_tot = s[..., 3] + 0 * n", 1)],
    "mean_cosine_not_divided_by_count": [
        (PY, "return s[..., 1] / s[..., 0]", "return s[..., 1] + 0 * s[..., 0]", 1)],
    # ridge fit
    "ridge_uncentred_normal_equations": [
        (C, "double xi = X[t * p + i] - xm[i];", "double xi = X[t * p + i];", 1),
        (C, "A[i * p + j] += xi * (X[t * p + j] - xm[j]);", "A[i * p + j] += xi * X[t * p + j];", 1)],
    "ridge_penalty_dropped": [(C, "A[i * p + i] += lam;", "A[i * p + i] += 0.0 * lam;", 1)],
    "ridge_penalty_scaled_by_n": [(C, "A[i * p + i] += lam;", "A[i * p + i] += lam * (double)n;", 1)],
    "ridge_intercept_sign": [
        (C, "v -= xm[i] * W[i * q + c];", "v += xm[i] * W[i * q + c];", 1)],
    "ridge_back_solve_with_L_not_LT": [
        (C, "v -= A[m * p + i] * W[m * q + c];", "v -= A[i * p + m] * W[m * q + c];", 1)],
    # layer-selection scores
    "scores_target_keys_not_unrotated": [
        (C, "if (m == 0) kvxo_rope(y, (int)d, (double)pos[g], P->theta_tgt, -1, Y + g * d);",
         "if (m == 0) memcpy(Y + g * d, y, sizeof(double) * (size_t)d);", 1)],
    "scores_source_keys_unrotated_with_target_base": [
        (C, "if (m == 0) kvxo_rope(x, (int)d, (double)pos[g], P->theta_src, -1, X + g * d);",
         "if (m == 0) kvxo_rope(x, (int)d, (double)pos[g], P->theta_tgt, -1, X + g * d);", 1)],
    "scores_total_uncentred": [
        (C, "double c = Y[g * d + i] - ym[i];", "double c = Y[g * d + i];", 1)],
    "scores_prediction_without_intercept": [
        (C, "double pred = b[i];", "double pred = 0.0 * b[i];", 1)],
    "scores_set_from_first_layer_only": [
        (C, "int64_t s = P->layer_idx[lt * k + j];\n              const double *x",
         "int64_t s = P->layer_idx[lt * k + 0];\n              const double *x", 1)],
    # ridge-fit inputs
    "features_keys_unrotated_with_target_base": [
        (C, "if (m == 0) kvxo_rope(v, (int)d, (double)p, P->theta_src, -1, o);",
         "if (m == 0) kvxo_rope(v, (int)d, (double)p, P->theta_tgt, -1, o);", 1)],
    "features_target_keys_left_rotated": [
        (C, "if (m == 0) kvxo_rope(v, (int)d, (double)p, P->theta_tgt, -1, o);",
         "if (m == 0) memcpy(o, v, sizeof(double) * (size_t)d);", 1)],
    "features_layers_side_by_side_in_reverse": [
        (C, "double *o = x + (b * ntok + g) * k * d + j * d;",
         "double *o = x + (b * ntok + g) * k * d + (k - 1 - j) * d;", 1)],
    "features_bad_layer_row_still_written": [
        (C, "for (int64_t j = 0; row_ok && j < k; ++j) {",
         "for (int64_t j = 0; (row_ok || P->layer_idx[lt * k + j] < Ls) && j < k; ++j) {", 1)],
}

# runs every pin function of test_oracle_pins (parametrized ones once per
# value) against the oracle package found first on sys.path
_CHILD = r"""
import json, sys
mut, tests, root = sys.argv[1:4]
sys.path[:0] = [mut, tests, root]
import pytest
import oracle
assert oracle.__file__.startswith(mut), oracle.__file__
import test_oracle_pins as T
passed, failed = 0, []
for name in sorted(vars(T)):
    fn = getattr(T, name)
    if not name.startswith("test_") or not callable(fn):
        continue
    calls = [{}]
    for m in getattr(fn, "pytestmark", []):
        if m.name == "parametrize":
            names = [a.strip() for a in m.args[0].split(",")]
            vals = [v if len(names) > 1 else (v,) for v in m.args[1]]
            calls = [dict(c, **dict(zip(names, v))) for c in calls for v in vals]
    for kw in calls:
        try:
            fn(**kw)
            passed += 1
        except (Exception, pytest.skip.Exception) as e:
            failed.append(f"{name}{kw or ''}: {type(e).__name__}")
print(json.dumps({"passed": passed, "failed": failed}))
"""


def _plant(tmp, name):
    dst = os.path.join(tmp, name, "oracle")
    os.makedirs(dst)
    for f in (PY, C, "kvx_oracle.h"):
        shutil.copy(os.path.join(ORACLE, f), os.path.join(dst, f))
    for f, old, new, count in MUTATIONS[name]:
        path = os.path.join(dst, f)
        text = open(path).read()
        assert text.count(old) == count, (name, old, text.count(old))
        open(path, "w").write(text.replace(old, new))
    return os.path.dirname(dst)


def _run(tmp, name):
    mut = _plant(tmp, name)
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    p = subprocess.run([sys.executable, "-c", _CHILD, mut, TESTS, ROOT], capture_output=True,
                       text=True, timeout=300, env=env)
    if p.returncode != 0:
        return {"crash": p.returncode, "stderr": p.stderr[-2000:]}
    return json.loads(p.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {n: ex.submit(_run, tmp, n) for n in MUTATIONS}
        return {n: f.result() for n, f in futs.items()}


def test_unchanged_copy_passes_every_pin(results):
    r = results["unchanged"]
    assert "crash" not in r, r
    assert r["failed"] == [] and r["passed"] >= 40, r


@pytest.mark.parametrize("name", [n for n in MUTATIONS if n != "unchanged"])
def test_planted_mistake_fails_a_pin(results, name):
    r = results[name]
    assert "crash" not in r, r
    assert r["failed"], f"no pin catches the planted mistake {name!r}"
