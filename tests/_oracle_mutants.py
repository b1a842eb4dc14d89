"""Planted mistakes in the oracle, used to show that its pins catch them.

Each mutant is one plausible slip in ``oracle/reference.py`` (a dropped term,
a wrong sign or index, a transposed operand, the other variance divisor...).
``apply(name)`` rewrites the oracle module in memory -- on the CPU, in the
test process only -- and ``test_oracle_mutants.py`` runs the oracle pin suite
under each mutant, expecting it to fail.
"""
import importlib
import inspect

# name -> (exact snippet in oracle/reference.py, its mutated replacement)
MUTANTS = {
    "attn_scale_dropped": ("* scale\n", "* 1.0\n"),
    "attn_causal_off_by_one": ("key_idx <= sel[:, None]", "key_idx < sel[:, None] + 2"),
    "attn_gqa_map_modulo": ("kvh = h // group", "kvh = h % Hkv"),
    "attn_k_for_v": ("acc = p @ v[b, kvh]", "acc = p @ k[b, kvh][:, :Dv]"),
    "attn_lse_missing_max": ("m_safe + np.log(l), NEG_INF", "np.log(l), NEG_INF"),
    "attn_not_normalised": ("acc / l[:, None]", "acc / l.max()"),
    "attn_exp_sign": ("p = np.exp(s - m_safe[:, None])", "p = np.exp(m_safe[:, None] - s)"),
    "split_bounds_overlap": ("((s + 1) * L) // num_splits)", "((s + 1) * L) // num_splits + 1)"),
    "merge_weight_not_normalised": ("np.exp(lse_part - np.where(live, lse, 0.0)[..., None])",
                                    "np.exp(lse_part - np.where(live, mx_safe, 0.0)[..., None])"),
    "merge_lse_missing_max": ("lse = np.where(live, mx_safe + np.log(total), NEG_INF)",
                              "lse = np.where(live, np.log(total), NEG_INF)"),
    "ln_unbiased_variance": ("keepdims=True) / n  # pass 2", "keepdims=True) / (n - 1)  # pass 2"),
    "ln_eps_outside_sqrt": ("np.sqrt(var + eps)", "(np.sqrt(var) + eps)"),
    "ln_residual_dropped": ("h = x + r ", "h = x + 0 * r "),
    "ln_beta_scaled": ("* g + b ", "* (g + b) "),
    "rms_mean_not_squared": ("ms = (h * h).sum(", "ms = (h * np.abs(h) * 0 + h).sum("),
    "rms_eps_outside_sqrt": ("np.sqrt(ms + eps) * g", "(np.sqrt(ms) + eps) * g"),
    "attn_window_off_by_one": ("s = np.where(key_idx > sel[:, None] - window, s, NEG_INF)",
                               "s = np.where(key_idx >= sel[:, None] - window, s, NEG_INF)"),
    "attn_alibi_sign": ("* (key_idx - sel[:, None])", "* (sel[:, None] - key_idx)"),
    "xent_target_sign": ("loss = np.where(valid, lse - tz, 0.0)", "loss = np.where(valid, lse + tz, 0.0)"),
    "xent_lse_missing_max": ("lse = (m + np.log(l))[..., 0]", "lse = (np.log(l))[..., 0]"),
    "xent_grad_no_onehot": ("t[valid]] -= 1.0", "t[valid]] -= 0.0"),
    "rms_residual_dropped": ("    h = x + r\n    n = h.shape[-1]\n    ms", "    h = x + 0 * r\n    n = h.shape[-1]\n    ms"),
    "rope_sin_sign": ("[x1 * c - x2 * s, x1 * s + x2 * c]", "[x1 * c + x2 * s, -x1 * s + x2 * c]"),
    "rope_interleaved_pairs": ("x1, x2 = x[..., :half], x[..., half:]", "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    "rope_frequency_exponent": ("** (-2.0 * np.arange(half, dtype=np.float64) / D)",
                                "** (-1.0 * np.arange(half, dtype=np.float64) / D)"),
}


def apply(name):
    import oracle
    import oracle.reference as ref

    old, new = MUTANTS[name]
    src = inspect.getsource(importlib.import_module("oracle.reference"))
    if src.count(old) != 1:
        raise RuntimeError(f"mutant {name}: snippet found {src.count(old)} times")
    code = compile(src.replace(old, new), ref.__file__, "exec")
    exec(code, ref.__dict__)
    for fn in ("attention", "decode", "decode_partials", "layernorm", "lse_merge", "split_bounds", "rmsnorm", "softmax_xent", "alibi_slopes", "rope"):
        setattr(oracle, fn, getattr(ref, fn))
