"""Each plausible mistake planted in a copy of the oracle trips at least one pin.

A mutant is the oracle source with one textual substitution (a dropped term,
a wrong sign or index, a swapped operand, a changed order) applied at every
place the text occurs (the same mistake made consistently), compiled with the
oracle's own flags into a temporary library.  The pins in oracle_pins.py run
against it; the test fails if all of them still pass.
"""
import os
import subprocess

import pytest

from oracle import zero1_oracle as o
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(o.__file__), "zero1_ref.c")

MUTANTS = {
    "decay_dropped": ("p = p * s->decay;", ";"),
    "decay_before_update": ("float p = master[i] - s->step_size * u;\n        p = p * s->decay;",
                            "float p = master[i] * s->decay;\n        p = p - s->step_size * u;"),
    "no_bias_correction": ("s->step_size = (float)(hp->lr * sqrt(bc2) / bc1);",
                           "s->step_size = (float)(hp->lr);"),
    "bias_betas_swapped": ("double bc1 = 1.0 - pow(hp->beta1, (double)t);\n    double bc2 = 1.0 - pow(hp->beta2, (double)t);",
                           "double bc1 = 1.0 - pow(hp->beta2, (double)t);\n    double bc2 = 1.0 - pow(hp->beta1, (double)t);"),
    "bias_exponent_off_by_one": ("pow(hp->beta1, (double)t)", "pow(hp->beta1, (double)t + 1.0)"),
    "eps_inside_sqrt": ("float d = sqrtf(vi) + s->eps;", "float d = sqrtf(vi + s->eps);"),
    "sum_not_mean": ("out[i] = s * inv_w;", "out[i] = s;"),
    "bf16_truncates": ("u += 0x7FFFu + lsb;", "(void)lsb;"),
    "bf16_ties_away": ("u += 0x7FFFu + lsb;", "(void)lsb; u += 0x8000u;"),
    "norm_without_sqrt": ("return sqrt(a->sum + a->comp);", "return a->sum + a->comp;"),
    "clip_inverted": ("if (norm > max_norm)\n        return (float)(max_norm / norm);",
                      "if (norm < max_norm)\n        return (float)(max_norm / norm);"),
    "clip_not_applied": ("float g = ghat[i] * c;", "float g = ghat[i];"),
    "clip_squared_norm": ("return (float)(max_norm / norm);", "return (float)(max_norm / (norm * norm));"),
    "rank_order_reversed": ("float s = zref_bf16_to_f32(grads[0][i]);\n        for (int q = 1; q < world; ++q)\n            s = s + zref_bf16_to_f32(grads[q][i]);",
                            "float s = zref_bf16_to_f32(grads[world - 1][i]);\n        for (int q = world - 2; q >= 0; --q)\n            s = s + zref_bf16_to_f32(grads[q][i]);"),
    "m_without_one_minus_beta1": ("mi = mi + s->one_minus_beta1 * g;", "mi = mi + g;"),
    "v_linear_in_g": ("vi = vi + og * g;", "vi = vi + og;"),
    "v_term_reassociated": ("vi = vi + og * g;", "vi = vi + s->one_minus_beta2 * (g * g); (void)og;"),
    "m_uses_beta2": ("float mi = s->beta1 * m[i];", "float mi = s->beta2 * m[i];"),
    "update_sign_flipped": ("float p = master[i] - s->step_size * u;", "float p = master[i] + s->step_size * u;"),
    "shard_drops_last_element": ("uint64_t a = (uint64_t)r * s, b = a + s;", "uint64_t a = (uint64_t)r * s, b = a + s - 1;"),
    "all_gather_one_replica": ("for (int q = 0; q < n_replicas; ++q) {", "for (int q = 0; q < 1; ++q) {"),
    "f32_allreduce_drops_last_rank": ("            for (int k = 1; k < world; ++k)\n                s = s + in[k][i];",
                                      "            for (int k = 1; k < world - 1; ++k)\n                s = s + in[k][i];"),
    "f32_allreduce_gather_wrong_slice": ("                out[q][i] = scratch[i];", "                out[q][i] = scratch[lo];"),
    "f32_allreduce_mean_ignored": ("            scratch[i] = average ? s * scale : s;", "            scratch[i] = s;"),
    "variant_decay_order_ignored": ("        if (o->decay_before_update) {", "        if (0) {"),
    "variant_clip_eps_ignored": ("    double q = max_norm / (norm + clip_eps);", "    double q = max_norm / norm;"),
    "variant_bf16_v_not_stored": ("            vb[i] = zref_f32_to_bf16(vi);", "            (void)vb;"),
    "variant_bf16_m_product_not_rounded": ("mi = bf16_round(s->beta1 * zref_bf16_to_f32(mb[i]));",
                                           "mi = s->beta1 * zref_bf16_to_f32(mb[i]);"),
    "variant_bf16_v_product_not_rounded": ("vi = bf16_round(s->beta2 * zref_bf16_to_f32(vb[i]));",
                                           "vi = s->beta2 * zref_bf16_to_f32(vb[i]);"),
    "variant_bf16_sqrt_not_rounded": ("d = bf16_round(bf16_round(sqrtf(vi)) + bf16_round(s->eps));",
                                      "d = bf16_round(sqrtf(vi) + bf16_round(s->eps));"),
    "variant_bf16_eps_not_rounded": ("d = bf16_round(bf16_round(sqrtf(vi)) + bf16_round(s->eps));",
                                     "d = bf16_round(bf16_round(sqrtf(vi)) + s->eps);"),
    "gather_shards_off_by_one": ("uint64_t lo = (uint64_t)r * shard_len, hi = lo + shard_len;",
                                 "uint64_t lo = (uint64_t)r * shard_len, hi = lo + shard_len - 1;"),
    "stage1_not_sharded": ("case 1: return (2.0 + 2.0) * psi + k * psi / w;", "case 1: return (2.0 + 2.0 + k) * psi;"),
    "ring_missing_factor": ("return op == 0 ? 2.0 * one : one;", "return one;"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def _catchers(name, source, tmp_path) -> list[str]:
    """The pins that fail on the oracle with mutant `name` planted."""
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *o.CFLAGS, "-o", str(so), str(src), "-lm"], check=True)
    prev = o.use(o.load(str(so)))
    caught = []
    try:
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(pin.__name__)
    finally:
        o.use(prev)
    return caught


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    assert _catchers(name, source, tmp_path), f"no pin caught the planted mistake {name}"


def test_second_moment_association_needs_the_inplace_ops_pin(source, tmp_path):
    """(1-b2)*(g*g) in place of ((1-b2)*g)*g stays within the 1e-6 parity
    tolerance and passes the closed forms and the float64 torch.optim.AdamW
    comparison; the page's in-place ops run by torch on fp32 tensors are
    what tell the two associations apart."""
    assert _catchers("v_term_reassociated", source, tmp_path) == ["pin_fp32_update_vs_torch_inplace_ops"]
