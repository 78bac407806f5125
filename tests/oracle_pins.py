"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a value printed on the pages, a closed form, an invariant
or a brute-force/library computation.  ``test_oracle_pins`` runs them on the
real oracle; ``test_oracle_mutants`` runs them on deliberately broken copies
and requires every mutant to be caught.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U = 2.0 ** -24  # fp32 unit roundoff


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """Library cross-check: torch's round-to-nearest-even fp32 -> bf16 cast."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, np.uint32) << 16).view(np.float32)


def rand_bf16(rng, shape, scale=1.0):
    return bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


class Cfg:
    def __init__(self, lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.0):
        self.lr, self.beta1, self.beta2, self.eps = lr, beta1, beta2, eps
        self.weight_decay, self.max_norm = weight_decay, max_norm


def cfg_struct(step, **kw):
    from oracle import adamw_cfg
    return adamw_cfg(Cfg(**kw), step)


# --------------------------------------------------------------------------- planner
def pin_plan_golden(orc):
    """Hand-derived layout of the 7-tensor plumbing case (tests/golden)."""
    g = golden("plan_tiny_P4_1MiB.json")
    p = orc.plan(g["sizes"], g["bucket_bytes"], g["P"])
    assert p["t_off"].tolist() == g["t_off"]
    assert p["t_bucket"].tolist() == g["t_bucket"]
    assert p["b_off"].tolist() == g["b_off"]
    assert p["b_len"].tolist() == g["b_len"]
    assert p["L"] == g["L"]


def check_plan_invariants(sizes, cap_bytes, P, p):
    """Properties that determine the greedy reverse-order plan uniquely."""
    n = len(sizes)
    cap = cap_bytes // 2
    slot = [(s + 7) // 8 * 8 for s in sizes]
    q = 16 * P
    nb = p["n_buckets"]
    assert len(p["b_off"]) == nb
    off = 0
    for b in range(nb):                       # contiguous, padded to 16P
        assert p["b_off"][b] == off
        assert p["b_len"][b] % q == 0
        off += p["b_len"][b]
    assert p["L"] == off
    order = list(range(n - 1, -1, -1))        # reverse compute order
    members = [[t for t in order if p["t_bucket"][t] == b] for b in range(nb)]
    flat = [t for b in range(nb) for t in members[b]]
    assert flat == order, "tensors must fill buckets last-to-first"
    for b in range(nb):
        cur = p["b_off"][b]
        for t in members[b]:
            assert p["t_off"][t] == cur and cur % 8 == 0
            cur += slot[t]
        used = cur - p["b_off"][b]
        assert p["b_len"][b] - used < q      # minimal padding
        nonzero = [t for t in members[b] if slot[t] > 0]
        if len(nonzero) > 1:
            assert used <= cap, "a multi-tensor bucket stays within the cap"
        if b + 1 < nb:                         # greedy: the next tensor did not fit
            nxt = members[b + 1][0]
            assert used > 0 and used + slot[nxt] > cap


def pin_plan_invariants(orc):
    rng = np.random.default_rng(7)
    cases = [([5, 0, 17, 64, 3], 64, 2), ([0, 0, 0], 1024, 4), ([100000], 16, 3),
             ([8] * 50, 96, 5), ([1], 2, 1)]
    for _ in range(40):
        n = int(rng.integers(1, 30))
        sizes = rng.integers(0, 5000, size=n).tolist()
        P = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        cap = int(rng.choice([16, 256, 4096, 20000]))
        cases.append((sizes, cap, P))
    for sizes, cap, P in cases:
        check_plan_invariants(sizes, cap, P, orc.plan(sizes, cap, P))


# --------------------------------------------------------------------------- ring
def pin_ring_ownership(orc):
    """Rank r contributes 10**r: after the reduce-scatter exactly one chunk per
    rank carries every contribution, and rank c holds chunk c ("Data Parallelism: From
    Parameter Server to Ring All-Reduce", sec. 5: each rank ends the reduce-scatter
    holding one chunk's complete sum)."""
    for P in range(2, 7):
        S = 3
        X = np.zeros((P, P * S), np.float32)
        for r in range(P):
            X[r, :] = 10.0 ** r
        full = sum(10.0 ** r for r in range(P))
        Y, _, _ = orc.ring_reduce_scatter(X)
        for r in range(P):
            full_chunks = [c for c in range(P) if np.all(Y[r, c * S:(c + 1) * S] == full)]
            assert full_chunks == [r], (P, r, full_chunks)


def pin_ring_order(orc):
    """The owner's sum of chunk c folds ranks c+1, c+2, ..., c (mod P) from the
    left: with 2**24 at rank c+1, -2**24 at rank c and 1.0 elsewhere, every +1
    is absorbed and the chunk sums to exactly 0."""
    for P in range(3, 9):
        S = 2
        X = np.ones((P, P * S), np.float32)
        for c in range(P):
            X[(c + 1) % P, c * S:(c + 1) * S] = 2.0 ** 24
            X[c, c * S:(c + 1) * S] = -(2.0 ** 24)
        Y, _, _ = orc.ring_reduce_scatter(X)
        for c in range(P):
            assert np.all(Y[c, c * S:(c + 1) * S] == 0.0), (P, c, Y[c])


def pin_ring_sum_exact(orc):
    """Owner sums against the exact sum within the fp32 bound (P-1)u sum|g|."""
    rng = np.random.default_rng(11)
    for P in (2, 3, 4, 5, 8, 16):
        S = 40
        g = rand_bf16(rng, (P, P * S), 1e-3)
        X = bf16_to_f32(g)
        Y, _, _ = orc.ring_reduce_scatter(X)
        exact = X.astype(np.float64).sum(0)
        bound = (P - 1) * U * np.abs(X.astype(np.float64)).sum(0) + 1e-45
        for c in range(P):
            sl = slice(c * S, (c + 1) * S)
            assert np.all(np.abs(Y[c, sl].astype(np.float64) - exact[sl]) <= bound[sl])


def pin_ring_traffic(orc):
    """Per-rank volume (N-1)M/N per phase, 2(N-1)/N*M in total, 2(N-1) steps
    ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 5 and 6; "4.1 Data parallelism in depth", sec. 5.2)."""
    for P in (1, 2, 3, 4, 8, 16):
        M = 8 * P * 3
        _, s1, k1 = orc.ring_reduce_scatter(np.zeros((P, M), np.float32))
        _, s2, k2 = orc.ring_all_gather(np.zeros((P, M), np.uint16))
        assert np.all(s1 == (P - 1) * M // P) and np.all(s2 == (P - 1) * M // P)
        assert np.all((s1 + s2) * P == 2 * (P - 1) * M)
        assert k1 + k2 == 2 * (P - 1)


def pin_ring_allgather_payload(orc):
    """After the all-gather every rank holds every owner's chunk."""
    for P in (2, 3, 5, 8):
        S = 4
        Y = np.zeros((P, P * S), np.uint16)
        for c in range(P):
            Y[c, c * S:(c + 1) * S] = 1000 + c
        out, _, _ = orc.ring_all_gather(Y)
        want = np.repeat(1000 + np.arange(P), S).astype(np.uint16)
        for r in range(P):
            assert np.array_equal(out[r], want)


def pin_stage_traffic(orc):
    """DDP, ZeRO-1 and ZeRO-2 each send 2(P-1)/P*M per rank, ZeRO-3 3(P-1)/P*M:
    1.5x ("Data Parallelism: DDP, ZeRO and FSDP", 'The three stages'; "4.1 Data parallelism in depth", sec. 8)."""
    g = golden("ledger_pages.json")["comm_per_step"]["value"]
    for P in (2, 4, 8, 16):
        M = 8 * P * 5
        vols = {}
        for stage, name in ((0, "DDP"), (1, "ZeRO-1"), (2, "ZeRO-2"), (3, "ZeRO-3")):
            sent, _ = orc.stage_traffic(stage, P, M)
            assert np.all(sent == sent[0])
            vols[name] = Fraction(int(sent[0]) * P, (P - 1) * M)
            assert vols[name] == g[name], (P, name, vols[name])
        assert vols["ZeRO-3"] / vols["DDP"] == Fraction(3, 2)


# --------------------------------------------------------------------------- ledger
def pin_ledger(orc):
    g = golden("ledger_pages.json")
    br = g["bytes_per_param_breakdown"]["value"]
    comp = (br["params_bf16"], br["grads_bf16"], br["master_fp32"], br["adam_m_fp32"],
            br["adam_v_fp32"])
    assert sum(comp) == br["total"] == 16
    for P in (1, 2, 4, 8, 16, 64):
        assert orc.ledger_bytes(0, 1.0, P, comp) == 16.0
        assert math.isclose(orc.ledger_bytes(1, 1.0, P, comp), 4 + 12 / P)
        assert math.isclose(orc.ledger_bytes(2, 1.0, P, comp), 2 + 14 / P)
        assert math.isclose(orc.ledger_bytes(3, 1.0, P, comp), 16 / P)
    w = g["worked_7B_N8"]
    got = {k: orc.ledger_bytes(s, w["psi"], w["P"], comp) / 1e9
           for k, s in (("DDP", 0), ("ZeRO-2", 2), ("ZeRO-3", 3))}
    assert round(got["DDP"]) == w["value_GB"]["DDP"]
    assert round(got["ZeRO-2"]) == w["value_GB"]["ZeRO-2"]     # 26.25 printed as ~26
    assert round(got["ZeRO-3"]) == w["value_GB"]["ZeRO-3"]
    w = g["worked_70B_replica"]
    assert math.isclose(orc.ledger_bytes(0, w["psi"], 1, comp) / 1e12, w["value_TB"])
    w = g["worked_3B_fsdp"]
    c3 = (2, 0, 0, 4, 4)
    assert math.isclose(orc.ledger_bytes(0, w["psi"], 1, c3) / 1e9, w["value_GB"]["total"])
    assert math.isclose(orc.ledger_bytes(3, w["psi"], w["P"], c3) / 1e9,
                        w["value_GB"]["sharded_per_gpu"])
    q = g["zero3_fit_question"]
    smallest = next(P for P in range(1, 1000) if orc.ledger_bytes(3, 70e9, P, comp) <= 80e9)
    assert smallest == q["answer_derived_here"]


# --------------------------------------------------------------------------- all-reduce
def _pack_ok(orc, sizes, cap, P, rng, scale=1e-3):
    n = sum(sizes)
    return rand_bf16(rng, (P, n), scale)


def pin_allreduce_identical(orc):
    """Identical replicas average to themselves (average, not sum: "4.1 Data parallelism in depth", sec. 2)."""
    rng = np.random.default_rng(3)
    sizes, cap = [13, 256, 1000, 7], 1024
    for P in (2, 3, 4, 8):
        one = rand_bf16(rng, (1, sum(sizes)), 1e-2)
        g = np.repeat(one, P, axis=0)
        out, mean, st = orc.allreduce_mean(sizes, cap, P, g)
        assert np.array_equal(out, g)
        assert np.array_equal(mean, bf16_to_f32(one[0]))
        assert st.replicas_equal == 1


def pin_allreduce_mean_exact(orc):
    rng = np.random.default_rng(5)
    for P, sizes, cap in ((4, [3, 1000, 655, 1311, 2621], 4096), (8, [77, 4096, 1, 900], 2048),
                          (5, [4000, 17, 333], 1000), (16, [31, 64, 129], 256)):
        g = _pack_ok(orc, sizes, cap, P, rng)
        out, mean, st = orc.allreduce_mean(sizes, cap, P, g)
        X = bf16_to_f32(g).astype(np.float64)
        exact = X.sum(0) / P
        bound = (P - 1) * U * np.abs(X).sum(0) / P + U * np.abs(exact) + 1e-45
        assert np.all(np.abs(mean - exact) <= bound)
        for r in range(P):
            assert np.array_equal(out[r], bf16_bits(mean))
        assert st.replicas_equal == 1
        p = orc.plan(sizes, cap, P)
        assert st.n_buckets == p["n_buckets"] and st.padded_len == p["L"]
        for r in range(P):   # ring volume over all buckets: 2(P-1)/P * L
            assert (st.rs_sent[r] + st.ag_sent[r]) * P == 2 * (P - 1) * p["L"]
        assert st.rs_steps + st.ag_steps == 2 * (P - 1) * p["n_buckets"]


def pin_bf16_rne(orc):
    cases = [1.0, -2.5, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, 3.4e38,
             1e-40, -0.0, 65504.0, 2.0 ** -133]
    hand = {1.0: 0x3F80, -2.5: 0xC020, 1.0 + 2 ** -8: 0x3F80, 1.0 + 3 * 2 ** -8: 0x3F82,
            1.0 + 2 ** -8 + 2 ** -20: 0x3F81}
    lib = bf16_bits(np.array(cases, np.float32))
    for x, want in zip(cases, lib):
        got = orc.bf16_rne(x)
        assert got == int(want), (x, hex(got), hex(int(want)))
        if x in hand:
            assert got == hand[x]
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000)).astype(np.float32)
    assert all(orc.bf16_rne(v) == int(w) for v, w in zip(x, bf16_bits(x)))


# --------------------------------------------------------------------------- AdamW
def pin_adamw_t1_closed_form(orc):
    """At t=1 the bias corrections give m_hat = g and v_hat = g*g, so
    theta1 = theta0 (1 - lr wd) - lr g / (|g| + eps)."""
    lr, wd, eps = 2e-4, 0.1, 1e-8
    for g in (1e-3, -5e-4, 3e-7, -2.0, 0.0):
        for decay in (0, 1):
            theta0 = 0.0173
            st = orc.adamw_element(g, theta0, 0.0, 0.0, decay, cfg_struct(1, lr=lr, weight_decay=wd))
            g32 = float(np.float32(g))
            want = theta0 * (1 - lr * wd * decay) - lr * g32 / (abs(g32) + eps)
            assert abs(st[0] - want) <= 8 * U * abs(theta0) + 1e-6 * lr, (g, decay, st[0], want)
            assert math.isclose(st[1], 0.1 * g32, rel_tol=4 * U, abs_tol=1e-45)
            assert math.isclose(st[2], 0.05 * g32 * g32, rel_tol=8 * U, abs_tol=1e-45)


def pin_adamw_weight_decay_only(orc):
    """Zero gradient: only decoupled decay acts, theta (1 - lr wd), exactly in fp32."""
    for step in (1, 2, 7):
        st = orc.adamw_element(0.0, 0.5, 0.0, 0.0, 1, cfg_struct(step, lr=1e-2, weight_decay=0.5))
        assert st[0] == np.float32(0.5) * np.float32(1 - 1e-2 * 0.5)
        st = orc.adamw_element(0.0, 0.5, 0.0, 0.0, 0, cfg_struct(step, lr=1e-2, weight_decay=0.5))
        assert st[0] == np.float32(0.5)


def pin_adamw_constant_gradient(orc):
    """With a constant gradient the bias-corrected moments are g and g*g at every
    step, so each step moves theta by lr g / (|g| + eps)."""
    lr, eps = 1e-3, 1e-8
    for g in (2e-3, -7e-5):
        theta, m, v = 0.25, 0.0, 0.0
        for t in range(1, 11):
            theta, m, v = orc.adamw_element(g, theta, m, v, 0,
                                            cfg_struct(t, lr=lr, weight_decay=0.0))
            g32 = float(np.float32(g))
            want = 0.25 - t * lr * g32 / (abs(g32) + eps)
            assert abs(theta - want) <= t * 1e-5 * lr + 4 * t * U * 0.25, (t, theta, want)


def pin_adamw_two_steps(orc):
    """Two different gradients: m2 = b1(1-b1)g1 + (1-b1)g2, v2 likewise with g^2,
    bias-corrected by 1-b^2 (the recurrence unrolled)."""
    b1, b2, lr, eps = 0.9, 0.95, 1e-3, 1e-8
    g1, g2, th = 3e-3, -1e-3, 0.1
    s = orc.adamw_element(g1, th, 0.0, 0.0, 0, cfg_struct(1, lr=lr, weight_decay=0.0))
    s = orc.adamw_element(g2, s[0], s[1], s[2], 0, cfg_struct(2, lr=lr, weight_decay=0.0))
    m2 = b1 * (1 - b1) * g1 + (1 - b1) * g2
    v2 = b2 * (1 - b2) * g1 * g1 + (1 - b2) * g2 * g2
    th1 = th - lr * g1 / (abs(g1) + eps)
    want = th1 - lr * (m2 / (1 - b1 ** 2)) / (math.sqrt(v2 / (1 - b2 ** 2)) + eps)
    assert math.isclose(s[1], m2, rel_tol=1e-6)
    assert math.isclose(s[2], v2, rel_tol=1e-6)
    assert abs(s[0] - want) <= 1e-5 * lr + 8 * U * th


# --------------------------------------------------------------------------- clip
def pin_clip_coef(orc):
    """clip_grad_norm_(params, 1.0) after averaging ("Distributed Training: Data Parallel, Model Parallel and FSDP Strategies", 'Inside DDP'):
    norm over all buckets, coef = min(1, max/(norm+1e-6)); library cross-check."""
    rng = np.random.default_rng(9)
    parts = rng.random(17) * 3.0
    coef, norm = orc.clip_coef(parts, 1.0)
    assert math.isclose(norm, math.sqrt(math.fsum(parts)), rel_tol=1e-15)
    assert math.isclose(coef, 1.0 / (norm + 1e-6), rel_tol=U)
    assert coef * norm <= 1.0 + 1e-6
    assert orc.clip_coef(np.array([0.25]), 1.0)[0] == 1.0          # norm 0.5 < 1
    assert orc.clip_coef(np.array([16.0]), 0.0)[0] == 1.0          # clipping off
    assert orc.clip_coef(np.array([16.0]), -1.0)[0] == 1.0
    # torch's clip_grad_norm_ on the same vector (fp32 norm): agree to ~1e-6
    vec = rng.standard_normal(5000).astype(np.float32) * 0.3
    t = torch.from_numpy(vec.copy()).requires_grad_()
    t.grad = torch.from_numpy(vec.copy())
    torch.nn.utils.clip_grad_norm_([t], 1.0)
    tcoef = float(t.grad[0] / t.grad.new_tensor(vec[0]))
    coef, _ = orc.clip_coef(np.array([float(np.sum(vec.astype(np.float64) ** 2))]), 1.0)
    assert math.isclose(coef, tcoef, rel_tol=2e-6)


def pin_norm_sum_is_exact(orc):
    """The clip norm is the 2-norm of the mean: one element of 1.0 followed by
    2**20 elements of 2**-27 gives sum(mean^2) = 1 + 2**-34 exactly, which a
    plain running double sum loses entirely (each 2**-54 is below half an ulp)."""
    n_small = 1 << 20
    sizes = [n_small, 1]                       # the 1-element tensor is packed first
    g = np.zeros((1, n_small + 1), np.uint16)
    g[0, :n_small] = bf16_bits(np.array([2.0 ** -27], np.float32))[0]
    g[0, n_small] = bf16_bits(np.array([1.0], np.float32))[0]
    sums = orc.bucket_sumsq(sizes, 1 << 30, 1, g)
    assert len(sums) == 1 and sums[0] == 1.0 + 2.0 ** -34, sums[0] - 1.0
    assert orc.sum(np.array([1.0] + [2.0 ** -54] * 1024)) == 1.0 + 2.0 ** -44


# --------------------------------------------------------------------------- fused step
def _zero_case(rng, P=4, sizes=(3, 1000, 655, 2621, 40), cap=4096, gscale=1e-3):
    sizes = list(sizes)
    n = sum(sizes)
    g = rand_bf16(rng, (P, n), gscale)
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    return sizes, cap, g, master


def pin_zero_step_t1(orc):
    """One fused step from m = v = 0 at t = 1 equals the closed form on the mean
    gradient, writes bf16(master) to every replica, and moves 2(P-1)/P*L."""
    rng = np.random.default_rng(21)
    for P in (2, 4, 8):
        sizes, cap, g, master = _zero_case(rng, P)
        decay = [1, 0, 1, 1, 0]
        n = sum(sizes)
        z = np.zeros(n, np.float32)
        lr, wd, eps = 2e-4, 0.1, 1e-8
        params, m2, mm, vv, mean, st = orc.zero_step(sizes, decay, cap, P, g, master, z, z,
                                                     cfg_struct(1, lr=lr, weight_decay=wd))
        X = bf16_to_f32(g).astype(np.float64)
        exact_mean = X.sum(0) / P
        assert np.all(np.abs(mean - exact_mean) <= (P - 1) * U * np.abs(X).sum(0) / P
                      + U * np.abs(exact_mean) + 1e-45)
        dflag = np.repeat(np.array(decay), sizes)
        gm = mean.astype(np.float64)
        want = master * (1 - lr * wd * dflag) - lr * gm / (np.abs(gm) + eps)
        assert np.all(np.abs(m2 - want) <= 8 * U * np.abs(master) + 1e-6 * lr)
        for r in range(P):
            assert np.array_equal(params[r], bf16_bits(m2))
        assert st.replicas_equal == 1 and st.coef == 1.0
        p = orc.plan(sizes, cap, P)
        for r in range(P):
            assert (st.rs_sent[r] + st.ag_sent[r]) * P == 2 * (P - 1) * p["L"]


def pin_zero_step_clip(orc):
    """Clipping acts on the averaged gradient: the norm is ||mean||_2 over all
    buckets and the update uses mean*coef."""
    rng = np.random.default_rng(23)
    P = 4
    sizes, cap, g, master = _zero_case(rng, P, gscale=5e-2)
    n = sum(sizes)
    z = np.zeros(n, np.float32)
    _, _, _, _, mean, st = orc.zero_step(sizes, [1] * 5, cap, P, g, master, z, z,
                                         cfg_struct(1, max_norm=1.0))
    norm = math.sqrt(math.fsum(mean.astype(np.float64) ** 2))
    assert norm > 1.0
    assert math.isclose(st.norm, norm, rel_tol=1e-12)
    assert math.isclose(st.coef, 1.0 / (norm + 1e-6), rel_tol=U)
    parts = orc.bucket_sumsq(sizes, cap, P, g)
    assert math.isclose(sum(parts), st.sumsq, rel_tol=1e-13)
    # the clipped step equals the unclipped step run on the pre-scaled mean,
    # checked at t=1 through the closed form theta0 - lr*gc/(|gc|+eps), gc = mean*coef
    _, m2, _, _, _, _ = orc.zero_step(sizes, [0] * 5, cap, P, g, master, z, z,
                                      cfg_struct(1, max_norm=1.0, weight_decay=0.0))
    gc = (mean * np.float32(st.coef)).astype(np.float64)
    want = master - 2e-4 * gc / (np.abs(gc) + 1e-8)
    assert np.all(np.abs(m2 - want) <= 8 * U * np.abs(master) + 1e-6 * 2e-4)


def pin_zero_vs_allreduce(orc):
    """Same reduce-scatter in both paths: identical fp32 means."""
    rng = np.random.default_rng(29)
    P = 8
    sizes, cap, g, master = _zero_case(rng, P)
    z = np.zeros(sum(sizes), np.float32)
    _, _, _, _, mz, _ = orc.zero_step(sizes, [1] * 5, cap, P, g, master, z, z, cfg_struct(1))
    _, ma, _ = orc.allreduce_mean(sizes, cap, P, g)
    assert np.array_equal(mz, ma)


def pin_zero_multi_step_state(orc):
    """State carries over: three steps equal three chained single-element updates
    on the same means (moments and step count advance)."""
    rng = np.random.default_rng(31)
    P = 4
    sizes, cap, _, master = _zero_case(rng, P)
    n = sum(sizes)
    mst, m, v = master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    ref = [(master[i], 0.0, 0.0) for i in (0, 5, 1500)]
    for t in (1, 2, 3):
        g = rand_bf16(rng, (P, n), 1e-3)
        _, mst, m, v, mean, _ = orc.zero_step(sizes, [1] * 5, cap, P, g, mst, m, v, cfg_struct(t))
        for k, i in enumerate((0, 5, 1500)):
            ref[k] = tuple(orc.adamw_element(mean[i], *ref[k], 1, cfg_struct(t)))
    for k, i in enumerate((0, 5, 1500)):
        assert (mst[i], m[i], v[i]) == tuple(np.float32(x) for x in ref[k])


# --------------------------------------------------------------------------- hybrid mesh
def pin_mesh_degenerate_equals_flat(orc):
    """An R x S mesh with R = 1 or S = 1 is the flat ring over P = R*S ranks."""
    rng = np.random.default_rng(41)
    sizes, cap = [13, 900, 2600, 77], 4096
    for P in (2, 4, 8):
        g = rand_bf16(rng, (P, sum(sizes)), 1e-3)
        flat, mflat, _ = orc.allreduce_mean(sizes, cap, P, g)
        for R, S in ((1, P), (P, 1)):
            out, mean, st = orc.mesh_allreduce_mean(sizes, cap, R, S, g)
            assert np.array_equal(out, flat) and np.array_equal(mean, mflat), (P, R, S)
            assert st.replicas_equal == 1


def pin_mesh_order(orc):
    """Hierarchical association: for shard 0 / sub-chunk 0 of a (2, 2) mesh the
    total is (g[1,1] + g[1,0]) + (g[0,1] + g[0,0]): with 2^24, 1, -2^24, 1 it is 1,
    where the flat ring's fold g1 + g2 + g3 + g0 gives 2."""
    P, R, S = 4, 2, 2
    n = 16 * P                                    # one bucket, shard = 32, sub-chunk = 16
    vals = {(1, 1): 2.0 ** 24, (1, 0): 1.0, (0, 1): -(2.0 ** 24), (0, 0): 1.0}
    X = np.zeros((P, n), np.float32)
    for (gi, si), val in vals.items():
        X[gi * S + si, :16] = val
    g16 = bf16_bits(X.ravel()).reshape(P, n)
    _, mean, _ = orc.mesh_allreduce_mean([n], 1 << 20, R, S, g16)
    _, mflat, _ = orc.allreduce_mean([n], 1 << 20, P, g16)
    assert mean[0] == 1.0 / P and mflat[0] == 2.0 / P


def pin_mesh_traffic(orc):
    """Per rank, per bucket of M elements: the in-group ring moves (S-1)/S*M twice,
    the cross-group all-reduce of one shard 2(R-1)/R * M/S; only the latter crosses
    groups ("4.1 Data parallelism in depth", sec. 5.2 ring volume, applied per level)."""
    rng = np.random.default_rng(43)
    for R, S in ((2, 4), (4, 2), (2, 2), (3, 2)):
        P = R * S
        M = 16 * P * 5
        g = rand_bf16(rng, (P, M), 1e-3)
        _, _, st = orc.mesh_allreduce_mean([M], 1 << 20, R, S, g)
        for r in range(P):
            assert Fraction(st.cross_sent[r]) == Fraction(2 * (R - 1) * M, R * S)
            assert Fraction(st.rs_sent[r] + st.ag_sent[r]) == \
                Fraction(2 * (S - 1) * M, S) + Fraction(2 * (R - 1) * M, R * S)
        flat_cross = Fraction(2 * (P - 1) * M, P)      # a flat ring over all P ranks
        assert Fraction(st.cross_sent[0]) < flat_cross


def pin_mesh_zero_step(orc):
    """Every group's owner of a shard applies the same update; all replicas equal;
    the (1, P) mesh is the flat step bit for bit, a (2, P/2) mesh within fp32
    reassociation of it."""
    rng = np.random.default_rng(47)
    P = 8
    sizes, cap, g, master = _zero_case(rng, P, sizes=(3, 1000, 655, 2621, 40), cap=4096)
    n = sum(sizes)
    z = np.zeros(n, np.float32)
    cfg = cfg_struct(1, max_norm=0.5)
    pf, mf, _, _, _, stf = orc.zero_step(sizes, [1] * 5, cap, P, g, master, z, z, cfg)
    p1, m1, _, _, st1 = orc.mesh_zero_step(sizes, [1] * 5, cap, 1, P, g, master, z, z, cfg)
    assert np.array_equal(p1, pf) and np.array_equal(m1, mf) and st1.coef == stf.coef
    p2, m2, _, _, st2 = orc.mesh_zero_step(sizes, [1] * 5, cap, 2, 4, g, master, z, z, cfg)
    assert st2.groups_equal == 1 and st2.replicas_equal == 1
    assert np.all(np.abs(m2 - mf) <= 1e-6 * np.abs(mf) + 1e-9)


# --------------------------------------------------------------------------- ZeRO-3
def pin_zero3_flow(orc):
    """ZeRO-3 moves 3(P-1)/P * M per rank (two all-gathers of the parameters and
    one reduce-scatter of the gradients: "Data Parallelism: DDP, ZeRO and FSDP",
    "The three stages"), every rank gathers exactly the shards' values, and the
    update equals the ZeRO-2 step's, since only where the parameters live differs."""
    rng = np.random.default_rng(53)
    for P in (2, 4, 8):
        sizes, cap, g, master = _zero_case(rng, P, sizes=(3, 1000, 655, 2621, 40), cap=4096)
        n = sum(sizes)
        z = np.zeros(n, np.float32)
        shards = bf16_bits(master)
        cfg = cfg_struct(1, max_norm=0.5)
        ps, m3, mm3, vv3, st = orc.zero3_step(sizes, [1, 0, 1, 1, 0], cap, P, g, shards, master, z,
                                              z, cfg)
        p2, m2, mm2, vv2, _, st2 = orc.zero_step(sizes, [1, 0, 1, 1, 0], cap, P, g, master, z, z,
                                                 cfg)
        assert st.gathered_ok == 1
        assert np.array_equal(m3, m2) and np.array_equal(mm3, mm2) and np.array_equal(vv3, vv2)
        assert np.array_equal(ps, p2[0]) and st.coef == st2.coef
        L = orc.plan(sizes, cap, P)["L"]
        for r in range(P):
            vol = st.ag_fwd_sent[r] + st.ag_bwd_sent[r] + st.rs_sent[r]
            assert Fraction(vol * P, (P - 1) * L) == 3
            assert st.ag_fwd_sent[r] == st.ag_bwd_sent[r] == st.rs_sent[r]


# --------------------------------------------------------------------------- accumulation / bf16 wire
def pin_accumulate(orc):
    """bf16 accumulation is fp32 add + round-to-nearest-even (torch's bf16 add
    as a library cross-check); small integers accumulate exactly."""
    rng = np.random.default_rng(59)
    a = rand_bf16(rng, (3, 4000), 1e-2)
    b = rand_bf16(rng, (3, 4000), 1e-2)
    got = orc.accumulate(a, b)
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    want = (ta + tb).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    ints = bf16_bits(np.arange(-50, 50, dtype=np.float32)).reshape(1, -1)
    assert np.array_equal(bf16_to_f32(orc.accumulate(ints, ints)), 2 * bf16_to_f32(ints))


def pin_bf16_wire(orc):
    """P = 2: one rounded add, the same as the fp32 reduction; P >= 3: bf16 partial
    sums absorb small terms (2^8 + 1 = 2^8 in bf16), bounded by (P-1) 2^-8 sum|g|."""
    rng = np.random.default_rng(61)
    sizes, cap = [1000, 333, 77], 4096
    g = rand_bf16(rng, (2, sum(sizes)), 1e-3)
    w, _ = orc.allreduce_mean_bf16wire(sizes, cap, 2, g)
    f, _, _ = orc.allreduce_mean(sizes, cap, 2, g)
    assert np.array_equal(w, f)
    P, n = 4, 64
    X = np.ones((P, n), np.float32)
    X[1, :] = 256.0                                     # first in the fold of chunk 0
    w, q = orc.allreduce_mean_bf16wire([n], 1 << 20, P, bf16_bits(X.ravel()).reshape(P, n))
    _, mf, _ = orc.allreduce_mean([n], 1 << 20, P, bf16_bits(X.ravel()).reshape(P, n))
    assert q[0] == 256.0 / P and mf[0] == 259.0 / P
    for P in (3, 5, 8):
        g = rand_bf16(rng, (P, sum(sizes)), 1e-3)
        _, q = orc.allreduce_mean_bf16wire(sizes, cap, P, g)
        Xd = bf16_to_f32(g).astype(np.float64)
        assert np.all(np.abs(q - Xd.sum(0) / P) <= (P - 1) * 2.0 ** -8 * np.abs(Xd).sum(0) / P
                      + 2.0 ** -24 * np.abs(q) + 1e-45)


# --------------------------------------------------------------------------- identity
def lsq_data():
    from workloads.gen import small_ints
    B, F = 64, 16
    x = np.array(small_ints(0, 1, B * F, -3, 3), np.float64).reshape(B, F)
    y = np.array(small_ints(0, 2, B, -5, 5), np.float64)
    th = np.array(small_ints(0, 3, F, -2, 2), np.float64)
    return x, y, th


def pin_lsq_identity(orc):
    """g_bar = (1/N) sum_k g_k equals the full-batch gradient for an equal split
    ("4.1 Data parallelism in depth", sec. 2); summing gives N g; an uneven split with per-shard means
    breaks the equality (sec. 2 note)."""
    x, y, th = lsq_data()
    g_full, g_k, g_bar, g_sum = orc.lsq_identity(x, y, th, [16, 16, 16, 16])
    # brute force in exact rationals
    res = [sum(Fraction(int(a)) * int(b) for a, b in zip(x[i], th)) - int(y[i]) for i in range(64)]
    exact = [sum(res[i] * int(x[i, f]) for i in range(64)) / 64 for f in range(16)]
    assert [Fraction(v) for v in g_full] == exact
    assert np.array_equal(g_bar, g_full)          # bit-exact in double
    assert np.array_equal(g_sum, 4 * g_full)
    _, _, g_bar_u, _ = orc.lsq_identity(x, y, th, [20, 12, 16, 16])
    assert not np.array_equal(g_bar_u, g_full)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
