"""Planted mistakes in the CPU oracle, for the mutation test.

Each mutant is one plausible error in one oracle function: a dropped term,
a wrong sign, index, axis or constant, a transposed operand, an off-by-one
range, a wrong tie rule.  It is given as (module, function, original
snippet, mutated snippet); ``apply`` recompiles that one function with the
snippet replaced, inside the oracle module's own namespace, so every caller
inside the oracle sees the mistake.  The original snippet must occur exactly
once in the function, so a mutant cannot silently stop applying when the
oracle changes.

Test infrastructure only: the mistake is planted in the oracle, on the CPU,
in a child pytest process (``test_oracle_mutants.py`` sets ORACLE_MUTANT and
``conftest.py`` calls ``apply`` before the pin tests are collected).  The
CUDA path is never involved.
"""
from __future__ import annotations

import importlib
import inspect
import textwrap

# name: (module, function, original, mutated[, statement run afterwards in
# the module namespace, for tables the module builds at import])
MUTANTS = {
    # ---- bf16 rounding and the router
    "bf16_round_7_bits": ("moe", "bf16_round", "np.maximum(e, -125) - 8", "np.maximum(e, -125) - 7"),
    "bf16_round_truncates": ("moe", "bf16_round", "np.rint(v[nz] / ulp)", "np.trunc(v[nz] / ulp)"),
    "topk_ties_to_higher_index": ("moe", "router_topk", "logits[t, e] > logits[t, best]",
                                  "logits[t, e] >= logits[t, best]"),
    "topk_softmax_over_all_experts": ("moe", "router_topk", "probs[t] = ex / ex.sum()",
                                      "probs[t] = ex / np.exp(logits[t] - sel.max()).sum()"),
    # ---- routing layout
    "offsets_floor_not_ceil": ("moe", "route_offsets", "(counts[e] + align - 1) // align * align",
                               "counts[e] // align * align"),
    "rank_reversed_in_expert": ("moe", "route_offsets", "r = int(demanded[e] + fill[e])",
                                "r = int(demanded[e] + counts[e] - 1 - fill[e])"),
    "overflow_off_by_one": ("moe", "route_offsets", "if true_total > M_cap:",
                            "if true_total >= M_cap:"),
    "offsets_not_clamped": ("moe", "route_offsets", "offsets = np.minimum(demanded, M_cap)",
                            "offsets = demanded.copy()"),
    # ---- permute, combine, router gradient
    "permute_row_of_pair_not_token": ("moe", "permute", "row = x[p // k]", "row = x[p % x.shape[0]]"),
    "permute_scale_by_token": ("moe", "permute", "np.asarray(scale).reshape(-1)[p]",
                               "np.asarray(scale).reshape(-1)[p // k]"),
    "combine_probs_slot_reversed": ("moe", "unpermute", "float(np.asarray(probs)[t, j])",
                                    "float(np.asarray(probs)[t, k - 1 - j])"),
    "router_grad_sign": ("moe", "router_grad", "dS[t, j] = float(dO[t] @ y_perm[r])",
                         "dS[t, j] = -float(dO[t] @ y_perm[r])"),
    # ---- gate/up interleaving and activations
    "interleave_gate_up_swapped": ("moe", "interleave_gate_up", "out[..., 0::2] = w_gate",
                                   "out[..., 0::2] = w_up"),
    "silu_drops_g": ("moe", "phi", "return g / (1.0 + np.exp(-g))",
                     "return 1.0 / (1.0 + np.exp(-g))"),
    "gelu_cubic_term_squared": ("moe", "phi", "0.5 * g * (1.0 + np.tanh(_C * (g + _A * g ** 3)))",
                                "0.5 * g * (1.0 + np.tanh(_C * (g + _A * g ** 2)))"),
    "dsilu_sign": ("moe", "dphi", "s * (1.0 + g * (1.0 - s))", "s * (1.0 - g * (1.0 - s))"),
    "dgelu_drops_3": ("moe", "dphi", "(1.0 + 3.0 * _A * g * g)", "(1.0 + _A * g * g)"),
    "srelu_not_squared": ("moe", "act_forward", "np.maximum(h, 0.0) ** 2", "np.maximum(h, 0.0)"),
    "gated_gate_up_swapped": ("moe", "act_forward", "phi(g, act) * u", "phi(u, act) * g"),
    "dgate_drops_u": ("moe", "act_backward", "dh[..., 0::2] = dA * u * dphi(g, act)",
                      "dh[..., 0::2] = dA * dphi(g, act)"),
    "dsrelu_drops_2": ("moe", "act_backward", "2.0 * np.maximum(h, 0.0) * dA",
                       "np.maximum(h, 0.0) * dA"),
    # ---- grouped MLP
    "fwd_fc2_wrong_expert": ("moe", "grouped_mlp_fwd", "_rb(a @ W2[e], round_bf16 and round_out)",
                             "_rb(a @ W2[0], round_bf16 and round_out)"),
    "fwd_drops_last_row_of_expert0": ("moe", "grouped_mlp_fwd",
                                      "r0, r1 = int(offsets[e]), int(offsets[e + 1])",
                                      "r0, r1 = int(offsets[e]), int(offsets[e + 1]) - (e == 0)"),
    "fwd_a_from_rounded_h_not_fc2_input": ("moe", "grouped_mlp_fwd",
                                           "Y[r0:r1] = _rb(a @ W2[e], round_bf16 and round_out)",
                                           "Y[r0:r1] = _rb(act_forward(h, act) @ W2[e], "
                                           "round_bf16 and round_out)"),
    "wgrad_operands_swapped": ("moe", "grouped_wgrad", "dW[e] = P[r0:r1].T @ Q[r0:r1]",
                               "dW[e] = (Q[r0:r1].T @ P[r0:r1]).reshape(dW[e].shape)"),
    "wgrad_drops_first_row": ("moe", "grouped_wgrad", "dW[e] = P[r0:r1].T @ Q[r0:r1]",
                              "dW[e] = P[r0 + 1:r1].T @ Q[r0 + 1:r1]"),
    "gemm_nk_not_transposed": ("moe", "grouped_gemm", "B = np.swapaxes(B, 1, 2)",
                               "B = B.reshape(B.shape[0], B.shape[2], B.shape[1])"),
    "bwd_dh_sign": ("moe", "grouped_mlp_bwd", "act_backward(H[r0:r1], dA, act)",
                    "act_backward(H[r0:r1], -dA, act)"),
    "bwd_dx_wrong_expert": ("moe", "grouped_mlp_bwd", "_rb(dh @ W1[e].T, round_bf16 and round_out)",
                            "_rb(dh @ W1[e - 1].T, round_bf16 and round_out)"),
    "bwd_dw2_transposed_product": ("moe", "grouped_mlp_bwd", "dW2[e] = A[r0:r1].T @ dY[r0:r1]",
                                   "dW2[e] = (dY[r0:r1].T @ A[r0:r1]).reshape(dW2[e].shape)"),
    "bwd_dw1_rows_shifted": ("moe", "grouped_mlp_bwd", "dW1[e] = x_perm[r0:r1].T @ dh",
                             "dW1[e] = x_perm[r0 + 1:r1 + 1].T @ dh"),
    "routed_drops_probability": ("moe", "grouped_mlp_bwd_routed",
                                 "act_backward(H[r0:r1], pr * dAp, act)",
                                 "act_backward(H[r0:r1], dAp, act)"),
    "routed_ds_scaled_twice": ("moe", "grouped_mlp_bwd_routed", "dS[r0:r1] = (dAp * A).sum(axis=1)",
                               "dS[r0:r1] = (pr * dAp * A).sum(axis=1)"),
    "routed_dw2_unscaled_a": ("moe", "grouped_mlp_bwd_routed", "dW2[e] = ap.T @ dO[r0:r1]",
                              "dW2[e] = A.T @ dO[r0:r1]"),
    # ---- NVFP4 statistics
    "hadamard_unnormalised": ("moe", "hadamard16", "/ 4.0", "/ 16.0"),
    "amax_without_abs": ("moe", "amax", "np.abs(t).max()", "t.max()"),
    "rht_rotation_dropped": ("moe", "amax_rht_transposed",
                             'rot = np.einsum("ij,bjc->bic", Hm, blk.reshape(nb, 16, G.shape[1]))',
                             "rot = blk.reshape(nb, 16, G.shape[1])"),
    "rht_blocks_not_from_expert_start": ("moe", "amax_rht_transposed", "blk[:rows] = G[r0:r1]",
                                         "blk[:rows] = G[r0 - r0 % 16:r0 - r0 % 16 + rows]"),
    # ---- MXFP8
    "e4m3_subnormal_exponent": ("mx", "e4m3_decode_table", "(m / 8.0) * 2.0 ** -6", "(m / 8.0) * 2.0 ** -7",
                                "_DEC = e4m3_decode_table(); _POS_VALS = _DEC[:0x7F]"),
    "e4m3_ties_to_odd": ("mx", "e4m3_encode", "np.where((hi & 1) == 0, hi, lo)",
                         "np.where((hi & 1) == 0, lo, hi)"),
    "e4m3_loses_negative_zero": ("mx", "e4m3_encode", "np.where(np.signbit(v.reshape(-1)), 0x80, 0)",
                                 "np.where(v.reshape(-1) < 0, 0x80, 0)"),
    "e8m0_emax_7": ("mx", "e8m0_exponent", "e = (ex - 1) - 8", "e = (ex - 1) - 7"),
    "e8m0_zero_block_unclamped": ("mx", "e8m0_exponent", "e = np.where(amax == 0, -127, e)", "e = e"),
    "weights_blocks_along_d": ("mx", "mx_quantize_weights",
                               "blk = W2.reshape(E, n // 32, 32, d).transpose(0, 1, 3, 2)",
                               "blk = W2.reshape(E, n, d // 32, 32).transpose(0, 2, 1, 3)"
                               ".reshape(E, n // 32, d, 32)"),
    "dequant_bias_128": ("mx", "mx_dequantize", "scale_codes.astype(np.int64) - 127",
                         "scale_codes.astype(np.int64) - 128"),
    "wgrad_drops_last_block": ("mx", "mx_wgrad", "dW[e] = P[:, r0:r1] @ Q[:, r0:r1].T",
                               "dW[e] = P[:, r0:r1 - 32] @ Q[:, r0:r1 - 32].T"),
    "mx_bwd_dw2_operands_swapped": ("mx", "mx_grouped_mlp_bwd",
                                    "mx_wgrad(a_qT, a_sT, dy_qT, dy_sT, offsets)",
                                    "mx_wgrad(dy_qT, dy_sT, a_qT, a_sT, offsets)"),
    "mx_bwd_dh_from_unscaled_w2": ("mx", "mx_grouped_mlp_bwd",
                                   "dA = mx_dgrad(dy_q, dy_s, w2_q, w2_s, offsets)",
                                   "dA = mx_dgrad(dy_q, dy_s, w2_q, np.full_like(w2_s, 127), offsets)"),
}


def apply(name: str) -> None:
    """Plant mutant ``name`` in the oracle package (this process only)."""
    import oracle
    mod_name, fn_name, old, new, *post = MUTANTS[name]
    mod = importlib.import_module(f"oracle.{mod_name}")
    src = textwrap.dedent(inspect.getsource(getattr(mod, fn_name)))
    n = src.count(old)
    if n != 1:
        raise RuntimeError(f"mutant {name}: snippet found {n} times in {mod_name}.{fn_name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    for stmt in post:
        exec(stmt, mod.__dict__)
    if hasattr(oracle, fn_name):
        setattr(oracle, fn_name, getattr(mod, fn_name))
    for attr in ("_DEC", "_POS_VALS"):
        if post and hasattr(oracle, attr):
            setattr(oracle, attr, getattr(mod, attr))
