"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source (a
dropped term, a wrong sign or index, a step out of order), builds it, swaps it
in for the real oracle and checks that at least one pin in test_oracle.py
fails. Everything runs on the CPU; the real oracle is restored afterwards.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTANTS = {
    "scalar_fade": ("Sh[(size_t)i * dv + j] *= a[i];", "Sh[(size_t)i * dv + j] *= a[0];"),
    "no_fade": ("Sh[(size_t)i * dv + j] *= a[i];", "(void)a;"),
    "error_sign": ("b * (v[tv + j] - u[j])", "b * (u[j] - v[tv + j])"),
    "no_beta": ("kn[i] * b * (v[tv + j] - u[j])", "kn[i] * (v[tv + j] - u[j])"),
    "predict_with_q": ("acc += kn[i] * Sh[(size_t)i * dv + j];\n                    u[j] = acc;",
                       "acc += qn[i] * Sh[(size_t)i * dv + j];\n                    u[j] = acc;"),
    "read_with_k": ("acc += qn[i] * Sh[(size_t)i * dv + j];\n                    o[tv + j]",
                    "acc += kn[i] * Sh[(size_t)i * dv + j];\n                    o[tv + j]"),
    "eps_outside_root": ("1.0 / sqrt(sq + eps)", "1.0 / (sqrt(sq) + eps)"),
    "scale_dropped": ("o[tv + j] = scale * acc;", "o[tv + j] = acc;"),
    "conv_taps_reversed": ("wc[0] * c0[c] + wc[1] * c1[c] + wc[2] * c2[c]\n                           + wc[3] * xt[c]",
                           "wc[3] * c0[c] + wc[2] * c1[c] + wc[1] * c2[c]\n                           + wc[0] * xt[c]"),
    "conv_no_silu": ("yt[c] = silu(pre);", "yt[c] = pre;"),
    "cache_not_shifted": ("c0[c] = c1[c];", "c0[c] = c0[c];"),
}

GATE_MUTANTS = {
    "gate_A_not_exponentiated": ("double z = exp(A_log[h]) *", "double z = A_log[h] *"),
    "gate_bias_dropped": ("(f[i] + dt_bias[(size_t)h * dk + c])", "(f[i])"),
    "gate_sign": ("double g = lb / (1.0 + exp(-z));", "double g = lb / (1.0 + exp(z));"),
    "gate_log_space": ("alpha[i] = exp(g);", "alpha[i] = g;"),
    "norm_sum_not_mean": ("sqrt(ss / dv + eps)", "sqrt(ss + eps)"),
    "norm_eps_outside_root": ("sqrt(ss / dv + eps)", "(sqrt(ss / dv) + eps)"),
    "norm_weight_dropped": ("oh[j] * r * w[j] /", "oh[j] * r /"),
    "norm_gate_not_sigmoid": ("/ (1.0 + exp(-gh[j]))", "* gh[j]"),
}

PINS = [
    pins.test_worked_example_states,
    pins.test_worked_example_reads,
    pins.test_worked_example_half_beta,
    lambda: pins.test_brute_force_dense_product(3, 8),
    lambda: pins.test_brute_force_dense_product(8, 3),
    pins.test_l2norm_eps_inside_root,
    pins.test_alpha1_beta0_leaves_state_and_reads_it,
    pins.test_beta1_unit_key_reads_back_value,
    pins.test_beta0_fades_each_row_by_its_alpha,
    pins.test_erase_shrinks_only_along_key,
    pins.test_scale_is_linear_on_output_only,
    pins.test_conv_identity_weights_is_silu,
    pins.test_conv_matches_direct_causal_convolution,
]


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + old
    bad = tmp_path / "mutant.c"
    bad.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", str(bad),
                           "-o", str(so), "-lm"])
    return oracle.bind(str(so))


@pytest.mark.parametrize("name", sorted(GATE_MUTANTS))
def test_gate_mutant_is_caught(name, tmp_path, monkeypatch):
    from tests import test_oracle_gate as gp
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, *GATE_MUTANTS[name]))
    caught = []
    for pin in (gp.test_gate_table_keep_factors_and_half_lives, gp.test_gate_neutral_point_and_floor,
                gp.test_gate_exp_A_scales_the_preactivation, gp.test_gate_bias_per_head_and_channel,
                gp.test_gate_range, gp.test_norm_constant_vector_and_open_gate,
                gp.test_norm_scale_invariance_and_unit_rms,
                gp.test_norm_gate_zero_halves_and_heads_independent, gp.test_norm_eps_inside_root):
        try:
            pin()
        except Exception:  # an assertion, or e.g. log of a negative "decay"
            caught.append(pin.__name__)
    assert caught, "no pin caught mutant " + name


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    bad = tmp_path / "mutant.c"
    bad.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", str(bad),
                           "-o", str(so), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.bind(str(so)))
    caught = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught.append(getattr(pin, "__name__", "pin"))
    assert caught, "no pin caught mutant " + name


def _tokens_variant(kind):
    """A copy of oracle.decode_tokens with one planted mistake."""
    import numpy as np

    def run(x, w, cache, alpha, beta, S0, scale=1.0, eps=oracle.L2_EPS):
        T = x.shape[1]
        S, c = np.array(S0, dtype=np.float64), np.array(cache, dtype=np.float64)
        o = np.empty(alpha.shape[:3] + (S.shape[-1],))
        order = range(T - 1, -1, -1) if kind == "reversed" else range(T)
        for t in order:
            ta = 0 if kind == "alpha_of_first" else t
            c_in = cache if kind == "cache_not_carried" else c
            S_in = S0 if kind == "state_not_carried" else S
            o[:, t], S, c = oracle.decode_step(x[:, t], w, c_in, alpha[:, ta], beta[:, t], S_in,
                                               scale=scale, eps=eps)
        return o, S, c
    return run


@pytest.mark.parametrize("kind", ["alpha_of_first", "cache_not_carried", "state_not_carried",
                                  "reversed"])
def test_tokens_mutant_is_caught(kind, monkeypatch):
    from tests import test_oracle_tokens as tp
    monkeypatch.setattr(oracle, "decode_tokens", _tokens_variant(kind))
    with pytest.raises(AssertionError):
        tp.test_tokens_equal_convolution_then_chunked_form(5)


# Planted mistakes in the chunked WY / UT form ("GLM-5.3 deep dive" 8.2.5,
# Eq. 6-9): each one replaces one line of a copy of oracle.chunk_prefill's
# source, and the pin that the chunked form reproduces the sequential
# recurrence must fail. (Keeping the diagonal in A is not among them: the
# forward substitution reads only A's strictly lower part, so that change
# computes the same thing.)
CHUNK_MUTANTS = {
    "exclusive_cumsum": ("G = np.cumsum(np.log(alpha[m, c0:c1, h]), axis=0)",
                         "G = np.cumsum(np.log(alpha[m, c0:c1, h]), axis=0)"
                         " - np.log(alpha[m, c0:c1, h])"),
    "Ki_grown_not_divided": ("Ki = K * np.exp(-G)", "Ki = K * np.exp(G)"),
    "A_without_beta": ("A = np.tril(b[:, None] * (Kd @ Ki.T), -1)",
                       "A = np.tril(Kd @ Ki.T, -1)"),
    "O_strictly_lower": ("np.tril(Qd @ Ki.T) @ Delta", "np.tril(Qd @ Ki.T, -1) @ Delta"),
    "beta_left_of_inverse": ("Mx = _unit_lower_solve(A, np.diag(b))",
                             "Mx = np.diag(b) @ _unit_lower_solve(A, np.eye(len(b)))"),
    "W_undecayed": ("W, U = Mx @ Kd, Mx @ V", "W, U = Mx @ K, Mx @ V"),
    "no_state_decay": ("Sh = np.exp(G[-1])[:, None] * Sh +", "Sh = Sh +"),
    "Kdec_from_chunk_start": ("(np.exp(G[-1] - G) * K).T", "(np.exp(-G) * K).T"),
}


@pytest.mark.parametrize("name", sorted(CHUNK_MUTANTS))
def test_chunked_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap
    old, new = CHUNK_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(oracle.chunk_prefill))
    assert src.count(old) == 1, "mutation site not found: " + name
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "chunk_prefill_mutant", "exec"), ns)
    monkeypatch.setattr(oracle, "chunk_prefill", ns["chunk_prefill"])
    with pytest.raises(AssertionError):
        pins.test_chunked_equals_sequential(65, 16)
