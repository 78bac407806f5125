"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one.  The mistakes are planted in the oracle, on the CPU: each
mutant is a textual edit of oracle.cpp compiled into a temporary library."""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "ring_direction": ("const int dst = (r + 1) % P;\n      const int c = mod(r - 1 - s, P);\n      float*",
                       "const int dst = (r + P - 1) % P;\n      const int c = mod(r - 1 - s, P);\n      float*"),
    "rs_schedule": ("const int c = mod(r - 1 - s, P);\n      std::memcpy(&msg",
                    "const int c = mod(r - s, P);\n      std::memcpy(&msg"),
    "ag_schedule": ("const int c = mod(r - s, P);\n      std::memcpy(&msg",
                    "const int c = mod(r - 1 - s, P);\n      std::memcpy(&msg"),
    "sum_not_mean": ("own[i] / static_cast<float>(P)", "own[i]"),
    "owner_shift": ("X.data() + static_cast<size_t>(c) * len + c * S;",
                    "X.data() + static_cast<size_t>((c + 1) % P) * len + c * S;"),
    "no_bias_correction1": ("c.lr / (1.0 - std::pow(c.beta1, t))", "c.lr"),
    "no_bias_correction2": ("std::sqrt(1.0 - std::pow(c.beta2, t))", "1.0"),
    "eps_inside_sqrt": ("std::sqrt(v) / s.sqrt_bc2 + s.eps", "std::sqrt(v + s.eps) / s.sqrt_bc2"),
    "decay_ignored": ("if (decay) theta = theta * s.wd_factor;", "(void)decay;"),
    "decay_coupled": ("if (decay) theta = theta * s.wd_factor;",
                      "if (decay) g = g + static_cast<float>(0.1) * theta;"),
    "betas_swapped": ("s.b1 = static_cast<float>(c.beta1);", "s.b1 = static_cast<float>(c.beta2);"),
    "v_linear_in_g": ("s.omb2 * (g * g)", "s.omb2 * g"),
    "update_sign": ("theta = theta - s.step_size * (m / denom);",
                    "theta = theta + s.step_size * (m / denom);"),
    "clip_no_min": ("std::min(1.0, max_norm / (norm + 1e-6))", "max_norm / (norm + 1e-6)"),
    "clip_on_sum": ("const float g = means[b][i] * coef;",
                    "const float g = means[b][i] * static_cast<float>(P) * coef;"),
    "plan_forward_order": ("for (int t = n - 1; t >= 0; --t) {\n    const int64_t slot",
                           "for (int t = 0; t < n; ++t) {\n    const int64_t slot"),
    "plan_pad_8": ("const int64_t quantum = 16 * static_cast<int64_t>(P);",
                   "const int64_t quantum = 8;"),
    "plan_pad_8P": ("const int64_t quantum = 16 * static_cast<int64_t>(P);",
                    "const int64_t quantum = 8 * static_cast<int64_t>(P);"),
    "norm_plain_sum": ("      comp += (sum - t) + x;\n    else\n      comp += (x - t) + sum;",
                       "      (void)0;\n    else\n      (void)0;"),
    "plan_close_ge": ("used + slot > cap", "used + slot >= cap"),
    "plan_no_align": ("const int64_t slot = (sizes[t] + 7) / 8 * 8;",
                      "const int64_t slot = sizes[t];"),
    "bf16_truncate": ("u += 0x7fffu + lsb;", "(void)lsb;"),
    "lsq_sum_not_mean": ("g_bar[f] = acc / N;", "g_bar[f] = acc;"),
    "ledger_zero2_keeps_grads": ("shard_grads = stage >= 2", "shard_grads = stage >= 3"),
    "mesh_rank_layout": ("X.data() + static_cast<size_t>(g * S + s) * len + s * sh, sizeof(float) * sh);",
                         "X.data() + static_cast<size_t>(s * R + g) * len + s * sh, sizeof(float) * sh);"),
    "mesh_no_cross_reduce": ("    ring_reduce_scatter(R, sh, C.data(), sent_rs, &steps);\n",
                             "    (void)sent_rs;\n"),
    "mesh_cross_ag_skipped": ("    ring_all_gather_f32(R, sh, C.data(), sent_ag, &steps);\n", "    (void)sent_ag;\n"),
    "zero3_fwd_gather_skipped": ("  for (int b = nb - 1; b >= 0; --b) gather(b, acc.ag_fwd_sent);     // forward",
                                 "  // forward gathers skipped"),
    "zero3_shard_not_updated": ("        param_shards[e] = f32_to_bf16_rne(master[e]);",
                                "        (void)e;"),
    "accumulate_sign": ("    acc[i] = f32_to_bf16_rne(bf16_bits_to_f32(acc[i]) + bf16_bits_to_f32(micro[i]));",
                        "    acc[i] = f32_to_bf16_rne(bf16_bits_to_f32(acc[i]) - bf16_bits_to_f32(micro[i]));"),
    "wire_receiver_overwrites": ("          mine[i] = f32_to_bf16_rne(bf16_bits_to_f32(mine[i]) + bf16_bits_to_f32(msg[static_cast<size_t>(r) * S + i]));",
                                 "          mine[i] = msg[static_cast<size_t>(r) * S + i];"),
    "zero3_one_gather": ("    ring_all_gather(P, M, Y.data(), sent, steps);\n    ring_all_gather(P, M, Y.data(), sent, steps);\n",
                         "    ring_all_gather(P, M, Y.data(), sent, steps);\n"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"oracle_{name}.cpp"
    src.write_text(source.replace(old, new))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.run(oracle.build_cmd(str(src), str(lib)), check=True)
    orc = oracle.Oracle(str(lib))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception as e:   # noqa: BLE001 - any failure counts as caught
            failed.append((pin.__name__, type(e).__name__))
    assert failed, f"mutant {name} passed every pin"
