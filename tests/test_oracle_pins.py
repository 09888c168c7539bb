"""Pins for the CPU oracle (no GPU): closed forms, hand-worked examples,
invariants, finite differences and torch library special cases. Each check is
independent of the oracle's own code path, so a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them
(test_planted_mistakes_are_caught plants some and checks exactly that)."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import coda_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def rand_block(M=3, d=8, f=8, seed=0, wscale=0.3):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((M, d)), z=rng.standard_normal((M, d)),
                W0=rng.standard_normal((d, d)) * wscale, W1=rng.standard_normal((d, 2 * f)) * wscale,
                W2=rng.standard_normal((f, d)) * wscale, gamma=rng.uniform(0.5, 1.5, d),
                dout=rng.standard_normal((M, d)))


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch_on_fp32_values():
    # torch's float32 -> bfloat16 conversion is round-to-nearest-even; on values
    # that are exact in fp32 the oracle's fp64 rounding must agree with it.
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_f16_round_matches_torch_and_ieee_binary16():
    # torch's float32 -> float16 conversion is IEEE round-to-nearest-even
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 12, 200000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(O.f16_round(v.astype(np.float64)), ref)
    ulp = 2.0 ** -10                                          # spacing of binary16 at 1
    assert O.f16_round(1 + ulp / 2) == 1.0                    # tie -> even (down)
    assert O.f16_round(1 + 3 * ulp / 2) == 1 + 2 * ulp        # tie -> even (up)
    assert O.f16_round(1 + ulp / 2 + 2 ** -30) == 1 + ulp
    assert O.f16_round(65504.0) == 65504.0                    # largest finite
    assert O.f16_round(65519.99) == 65504.0
    assert np.isinf(O.f16_round(65520.0))                     # rounds past the top
    assert O.f16_round(2.0 ** -24) == 2.0 ** -24              # smallest subnormal
    assert O.f16_round(2.0 ** -26) == 0.0


def test_saved_copies_are_fp16_rounded_in_the_storage_form():
    inp = rand_block(M=4, d=16, f=8, seed=9)
    fr = O.mlp_fwd_reparam(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"],
                           store_bf16=True)
    fe = O.mlp_fwd_reparam(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    assert np.array_equal(fr["y"], O.f16_round(fr["y"]))
    assert not np.array_equal(fe["y"], O.f16_round(fe["y"]))
    assert rel(fr["y"], fe["y"]) < 2.0 ** -11 * 1.01 + 1e-2  # hg's bf16 rounding dominates


def test_bf16_round_ties_to_even_and_nearest():
    one = 1.0
    ulp = 2.0 ** -7
    assert O.bf16_round(one + ulp / 2) == one                 # tie -> even (down)
    assert O.bf16_round(one + 3 * ulp / 2) == one + 2 * ulp   # tie -> even (up)
    assert O.bf16_round(one + ulp / 2 + 2 ** -30) == one + ulp
    assert O.bf16_round(-(one + ulp / 2 + 2 ** -30)) == -(one + ulp)
    # nearest: no other bf16 neighbour is closer
    rng = np.random.default_rng(2)
    x = rng.standard_normal(10000) * 7.3
    r = O.bf16_round(x)
    e = np.floor(np.log2(np.abs(r)))
    step = 2.0 ** (e - 7)
    assert np.all(np.abs(x - r) <= step / 2 * (1 + 1e-12) + 1e-300)


# ---------------------------------------------------------------- elementwise

def test_silu_closed_forms():
    for k, v in GOLD["silu"].items():
        assert abs(O.silu(float(k)) - v) < 1e-15
    for k, v in GOLD["dsilu"].items():
        assert abs(O.silu_grad(float(k)) - v) < 1e-15
    assert O.silu(0.0) == 0.0


def test_silu_grad_finite_difference():
    t = np.linspace(-8, 8, 101)
    hstep = 1e-6
    fd = (O.silu(t + hstep) - O.silu(t - hstep)) / (2 * hstep)
    assert np.max(np.abs(fd - O.silu_grad(t))) < 1e-8


def test_silu_matches_torch():
    t = np.linspace(-20, 20, 4001)
    assert rel(O.silu(t), F.silu(torch.from_numpy(t)).numpy()) < 1e-15


# ---------------------------------------------------------------- MLP block

def test_block_worked_example():
    g = GOLD["block_example"]
    i = g["inputs"]
    arr = lambda k: np.array(i[k], dtype=np.float64)
    x, z = arr("x")[None, :], arr("z")[None, :]
    fw = O.mlp_fwd(x, z, arr("W0"), arr("W1"), arr("W2"), arr("gamma"), eps=i["eps"])
    assert rel(fw["h"][0], g["h"]) < 1e-15
    assert abs(fw["r"][0] - g["r"]) < 1e-15
    assert rel(fw["y"][0], g["y"]) < 1e-14
    assert abs(fw["a"][0, 0] - g["a"]) < 1e-15
    assert rel(fw["out"][0], g["out"]) < 1e-14
    bw = O.mlp_bwd(fw, x, arr("W0"), arr("W1"), arr("W2"), arr("gamma"), arr("dout")[None, :])
    assert abs(bw["s"][0] - g["s"]) < 1e-14
    assert rel(bw["dy"][0], g["dy"]) < 1e-14
    assert rel(bw["dh"][0], g["dh"]) < 1e-13
    assert rel(bw["dgamma"], g["dgamma"]) < 1e-14
    assert rel(bw["dW0"], g["dW0"]) < 1e-13
    assert rel(bw["dW1"], g["dW1"]) < 1e-14
    assert rel(bw["dW2"], g["dW2"]) < 1e-14


def test_rms_factor_special_case_identity_weights():
    # W0 = I, z = 0: h = x, so r = 1/sqrt(mean(x^2) + eps) with eps inside the sqrt.
    rng = np.random.default_rng(3)
    d = 16
    x = rng.standard_normal((5, d))
    fw = O.mlp_fwd(x, np.zeros_like(x), np.eye(d), rng.standard_normal((d, 8)),
                   rng.standard_normal((4, d)), np.ones(d), eps=1e-6)
    for m in range(5):
        want = 1.0 / math.sqrt(sum(v * v for v in x[m]) / d + 1e-6)
        assert abs(fw["r"][m] - want) < 1e-15 * want
    # and with gamma = 1 the normalised rows have mean square mean/(mean+eps)
    ms = np.mean(fw["h2"] ** 2, axis=1)
    mx = np.mean(x * x, axis=1)
    assert np.allclose(ms, mx / (mx + 1e-6), rtol=1e-14)


def test_swiglu_zero_gate_and_limits():
    y = np.zeros((2, 8))
    y[:, 1::2] = 5.0
    assert np.all(O.swiglu(y) == 0.0)            # g = 0 -> a = 0 whatever u is
    y = np.zeros((1, 2))
    y[0] = [40.0, 2.0]                           # silu(40) = 40 to fp64 precision
    assert abs(O.swiglu(y)[0, 0] - 80.0) < 1e-12
    y[0] = [-40.0, 2.0]
    assert abs(O.swiglu(y)[0, 0]) < 1e-15


def _block_torch(inp, eps=1e-6):
    """Library special case: torch fp64 composition of rms_norm, silu and
    matmul, differentiated by autograd."""
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=k != "dout") for k, v in inp.items()}
    h = t["x"] @ t["W0"] + t["z"]
    h2 = F.rms_norm(h, (h.shape[1],), t["gamma"], eps)
    y = h2 @ t["W1"]
    a = F.silu(y[:, 0::2]) * y[:, 1::2]
    out = a @ t["W2"]
    (out * t["dout"]).sum().backward()
    return out.detach().numpy(), {k: t[k].grad.numpy() for k in ("x", "z", "W0", "W1", "W2", "gamma")}


def test_block_matches_torch_autograd():
    inp = rand_block(M=5, d=16, f=12, seed=4)
    out_t, grads_t = _block_torch(inp)
    fw = O.mlp_fwd(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    bw = O.mlp_bwd(fw, inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["dout"])
    assert rel(fw["out"], out_t) < 1e-13
    names = {"x": "dx", "z": "dz", "W0": "dW0", "W1": "dW1", "W2": "dW2", "gamma": "dgamma"}
    for k, v in names.items():
        assert rel(bw[v], grads_t[k]) < 1e-12, k


def fd_block_error(inp, step=1e-6):
    """Largest relative error, over every input, between the oracle's
    gradients and central finite differences of L = sum(dout * out)."""
    keys = ("x", "z", "W0", "W1", "W2", "gamma")

    def loss(vals):
        fw = O.mlp_fwd(vals["x"], vals["z"], vals["W0"], vals["W1"], vals["W2"], vals["gamma"])
        return float(np.sum(fw["out"] * inp["dout"]))

    fw = O.mlp_fwd(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    bw = O.mlp_bwd(fw, inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["dout"])
    gname = {"x": "dx", "z": "dz", "W0": "dW0", "W1": "dW1", "W2": "dW2", "gamma": "dgamma"}
    worst = 0.0
    for k in keys:
        base = inp[k]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            vals = {kk: inp[kk].copy() for kk in keys}
            vals[k][idx] += step
            lp = loss(vals)
            vals[k][idx] -= 2 * step
            lm = loss(vals)
            fd[idx] = (lp - lm) / (2 * step)
        worst = max(worst, rel(bw[gname[k]], fd))
    return worst


def test_block_backward_finite_differences():
    inp = rand_block(M=2, d=8, f=8, seed=5)
    assert fd_block_error(inp) < 1e-6


def test_reparam_equals_canonical():
    # commutation: r((xW0+z)*gamma)W1 = r(((xW0+z)*gamma)W1)  (exact arithmetic)
    inp = rand_block(M=7, d=24, f=16, seed=6)
    fc = O.mlp_fwd(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    fr = O.mlp_fwd_reparam(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    for k in ("h", "r", "y", "a", "out"):
        assert rel(fr[k], fc[k]) < 1e-12, k
    assert rel(fr["hg"] * fr["r"][:, None], fc["h2"]) < 1e-13
    bc = O.mlp_bwd(fc, inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["dout"])
    br = O.mlp_bwd_reparam(fr, inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["dout"])
    for k in ("s", "dh", "dx", "dW0", "dW1", "dW2", "dgamma"):
        assert rel(br[k], bc[k]) < 1e-11, k


def test_s_two_forms_agree():
    # s = (1/d) sumcols(dh2 * h2) = (1/d) sumcols(dy * y)  (notes s3)
    inp = rand_block(M=6, d=20, f=10, seed=7)
    fc = O.mlp_fwd(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    bc = O.mlp_bwd(fc, inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["dout"])
    d = inp["x"].shape[1]
    s1 = np.sum(bc["dh2"] * fc["h2"], axis=1) / d
    s2 = np.sum(bc["dy"] * fc["y"], axis=1) / d
    assert rel(s1, s2) < 1e-12
    assert rel(bc["s"], s1) < 1e-12


def test_storage_rounded_mode_rounds_stored_tensors_only():
    inp = rand_block(M=4, d=16, f=8, seed=8)
    fr = O.mlp_fwd_reparam(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"],
                           store_bf16=True)
    for k in ("h", "hg", "a", "out"):
        assert np.array_equal(fr[k], O.bf16_round(fr[k])), k
    fe = O.mlp_fwd_reparam(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    assert rel(fr["r"], fe["r"]) < 1e-15          # statistics come from the unrounded h
    assert rel(fr["out"], fe["out"]) < 2e-2


def rand_ln_block(M=3, d=8, f=8, seed=30):
    inp = rand_block(M, d, f, seed)
    inp["beta"] = np.random.default_rng(seed + 1).standard_normal(d) * 0.3
    return inp


def test_ln_block_matches_torch_layer_norm_and_autograd():
    inp = rand_ln_block(M=5, d=16, f=12, seed=31)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=k != "dout") for k, v in inp.items()}
    h = t["x"] @ t["W0"] + t["z"]
    h2 = F.layer_norm(h, (16,), t["gamma"], t["beta"], 1e-6)
    y = h2 @ t["W1"]
    out = (F.silu(y[:, 0::2]) * y[:, 1::2]) @ t["W2"]
    (out * t["dout"]).sum().backward()
    args = [inp[k] for k in ("x", "z", "W0", "W1", "W2", "gamma", "beta")]
    fw = O.ln_mlp_fwd(*args)
    bw = O.ln_mlp_bwd(fw, inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["beta"],
                      inp["dout"])
    assert rel(fw["out"], out.detach().numpy()) < 1e-13
    for k, g in (("x", "dx"), ("z", "dz"), ("W0", "dW0"), ("W1", "dW1"), ("W2", "dW2"),
                 ("gamma", "dgamma"), ("beta", "dbeta")):
        assert rel(bw[g], t[k].grad.numpy()) < 1e-12, k


def test_ln_block_finite_differences():
    inp = rand_ln_block(M=2, d=6, f=4, seed=32)
    keys = ("x", "z", "W0", "W1", "W2", "gamma", "beta")

    def L(v):
        return float(np.sum(O.ln_mlp_fwd(*[v[k] for k in keys])["out"] * inp["dout"]))

    fw = O.ln_mlp_fwd(*[inp[k] for k in keys])
    bw = O.ln_mlp_bwd(fw, inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["beta"],
                      inp["dout"])
    for k, gname in zip(keys, ("dx", "dz", "dW0", "dW1", "dW2", "dgamma", "dbeta")):
        fd = np.zeros_like(inp[k])
        for idx in np.ndindex(inp[k].shape):
            v = {kk: np.array(inp[kk], copy=True) for kk in keys}
            v[k][idx] += 1e-6
            lp = L(v)
            v[k][idx] -= 2e-6
            fd[idx] = (lp - L(v)) / 2e-6
        assert rel(bw[gname], fd) < 1e-6, k


def test_ln_reparam_equals_canonical():
    inp = rand_ln_block(M=7, d=24, f=16, seed=33)
    args = [inp[k] for k in ("x", "z", "W0", "W1", "W2", "gamma", "beta")]
    fc = O.ln_mlp_fwd(*args)
    fr = O.ln_mlp_fwd_reparam(*args)
    for k in ("mu", "r", "y", "a", "out"):
        assert rel(fr[k], fc[k]) < 1e-12, k
    bargs = (inp["x"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], inp["beta"], inp["dout"])
    bc = O.ln_mlp_bwd(fc, *bargs)
    br = O.ln_mlp_bwd_reparam(fr, *bargs)
    for k in ("sa", "sb", "dh", "dx", "dW0", "dW1", "dW2", "dgamma", "dbeta"):
        assert rel(br[k], bc[k]) < 1e-11, k
    assert rel(br["hhat"] * fr["r"][:, None], fc["h2"]) < 1e-12
    frs = O.ln_mlp_fwd_reparam(*args, store_bf16=True)
    for k in ("h", "hg", "a", "out"):
        assert np.array_equal(frs[k], O.bf16_round(frs[k])), k


def test_ln_with_zero_mean_rows_reduces_to_rmsnorm():
    # rows whose h has zero mean and beta = 0: LayerNorm equals RMSNorm
    inp = rand_block(M=4, d=8, f=6, seed=34)
    inp["W0"] = np.eye(8)
    inp["z"] = np.zeros((4, 8))
    inp["x"] = inp["x"] - inp["x"].mean(1, keepdims=True)
    ln = O.ln_mlp_fwd(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"], np.zeros(8))
    rm = O.mlp_fwd(inp["x"], inp["z"], inp["W0"], inp["W1"], inp["W2"], inp["gamma"])
    assert rel(ln["out"], rm["out"]) < 1e-13


# ---------------------------------------------------------------- cross-entropy

def test_ce_zero_weights_closed_form():
    V = 128256
    hidden = np.random.default_rng(9).standard_normal((2, 4))
    res = O.lmhead_ce(hidden, np.zeros((4, V)), np.array([0, V - 1]))
    assert np.allclose(res["lse"], GOLD["ln_V_128256"], rtol=0, atol=1e-12)
    assert np.allclose(res["loss"], GOLD["ln_V_128256"], rtol=0, atol=1e-12)


def test_ce_small_closed_form():
    W = np.array([[0.0, math.log(2), math.log(3), 0.0]])
    res = O.lmhead_ce(np.ones((2, 1)), W, np.array([2, 0]))
    g = GOLD["ce_small"]
    assert abs(res["lse"][0] - g["lse"]) < 1e-15
    assert abs(res["loss"][0] - g["loss_target2"]) < 1e-15
    assert abs(res["loss"][1] - g["loss_target0"]) < 1e-15


def test_ce_exact8_closed_form():
    g = GOLD["ce_exact8"]
    W = np.array([g["logits"]])
    res = O.lmhead_ce(np.ones((8, 1)), W, np.arange(8))
    assert np.allclose(res["lse"], g["lse"], rtol=0, atol=1e-14)
    assert np.allclose(res["loss"], g["loss"], rtol=0, atol=1e-14)


def test_ce_brute_force_and_torch():
    rng = np.random.default_rng(10)
    hidden = rng.standard_normal((6, 5))
    W = rng.standard_normal((5, 37)) * 2.0
    t = rng.integers(0, 37, 6)
    res = O.lmhead_ce(hidden, W, t)
    for i in range(6):
        logits = [sum(hidden[i, k] * W[k, j] for k in range(5)) for j in range(37)]
        lse = math.log(sum(math.exp(v) for v in logits))
        assert abs(res["lse"][i] - lse) < 1e-12
        assert abs(res["loss"][i] - (lse - logits[t[i]])) < 1e-12
    ref = F.cross_entropy(torch.from_numpy(hidden @ W), torch.from_numpy(t), reduction="none")
    assert rel(res["loss"], ref.numpy()) < 1e-13
    assert rel(res["lse"], torch.logsumexp(torch.from_numpy(hidden @ W), 1).numpy()) < 1e-14


def test_ce_large_logits_no_overflow():
    hidden = np.array([[1000.0], [-1000.0]])
    W = np.array([[1.0, 0.5, -2.0]])
    res = O.lmhead_ce(hidden, W, np.array([0, 2]))
    # row 0: logits 1000, 500, -2000 -> lse = 1000 + log(1 + e^-500 + ...) = 1000
    assert abs(res["lse"][0] - 1000.0) < 1e-12 and res["loss"][0] < 1e-12
    assert abs(res["lse"][1] - 2000.0) < 1e-12 and abs(res["loss"][1]) < 1e-12


def test_lse_two_level_equals_definition():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((9, 1000)) * 6
    direct = np.log(np.sum(np.exp(logits), axis=1))
    for tile in (1, 7, 128, 256, 999, 1000, 4096):
        assert rel(O.lse_two_level(logits, tile), direct) < 1e-14
    # shift invariance: adding c_i to row i adds c_i to the LSE
    c = rng.standard_normal(9) * 100
    assert rel(O.lse_two_level(logits + c[:, None], 100) - c, direct) < 1e-12


def test_ce_backward_finite_differences_and_torch():
    rng = np.random.default_rng(19)
    M, d, V = 4, 6, 11
    hidden = rng.standard_normal((M, d))
    W = rng.standard_normal((d, V)) * 0.7
    t = rng.integers(0, V, M)
    dloss = rng.standard_normal(M)
    res = O.lmhead_ce_bwd(hidden, W, t, dloss)

    def L(h, w):
        return float(np.sum(dloss * O.lmhead_ce(h, w, t)["loss"]))

    for name, X in (("dhidden", hidden), ("dW", W)):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp = X.copy(); Xp[idx] += 1e-6
            Xm = X.copy(); Xm[idx] -= 1e-6
            args_p = (Xp, W) if name == "dhidden" else (hidden, Xp)
            args_m = (Xm, W) if name == "dhidden" else (hidden, Xm)
            fd[idx] = (L(*args_p) - L(*args_m)) / 2e-6
        assert rel(res[name], fd) < 1e-6, name
    th = torch.tensor(hidden, requires_grad=True)
    tw = torch.tensor(W, requires_grad=True)
    loss = F.cross_entropy(th @ tw, torch.from_numpy(t), reduction="none")
    (loss * torch.from_numpy(dloss)).sum().backward()
    assert rel(res["dhidden"], th.grad.numpy()) < 1e-13
    assert rel(res["dW"], tw.grad.numpy()) < 1e-13
    # each row of G sums to zero (softmax sums to one, so does the one-hot row)
    assert np.max(np.abs(res["G"].sum(1))) < 1e-14


def test_ce_backward_columns_match_full_form():
    rng = np.random.default_rng(20)
    M, d, V = 7, 5, 300
    hidden = rng.standard_normal((M, d))
    W = rng.standard_normal((d, V))
    t = rng.integers(0, V, M)
    dloss = rng.standard_normal(M)
    full = O.lmhead_ce_bwd(hidden, W, t, dloss)["dW"]
    cols = np.array([0, 1, 17, t[0], 299])
    for chunk in (7, 64, 300, 1000):
        assert rel(O.lmhead_ce_dW_columns(hidden, W, t, dloss, cols, chunk), full[:, cols]) < 1e-13


# ---------------------------------------------------------------- RoPE

def test_rope_frequencies_closed_form():
    f = O.rope_inv_freq(128, 500000.0)
    for i, v in GOLD["rope_inv_freq_5e5_128"].items():
        assert abs(f[int(i)] - v) <= 1e-15 * max(v, 1e-300) * 4
    assert f[0] == 1.0


def test_rope_small_closed_form():
    v = np.array([[1.0, 0.0, 0.0, 1.0]])
    out = O.rope_apply(v, np.array([3]), n_rope_cols=4, head_dim=4, theta=10000.0)
    assert rel(out[0], GOLD["rope_hd4_pos3"]) < 1e-15


def test_rope_invariants():
    rng = np.random.default_rng(12)
    hd, nrope, ncols = 16, 48, 64
    v = rng.standard_normal((10, ncols))
    pos = rng.integers(0, 4096, 10)
    r = O.rope_apply(v, pos, nrope, hd, 500000.0)
    assert np.array_equal(r[:, nrope:], v[:, nrope:])                       # v columns untouched
    pn = lambda a: a[:, 0:nrope:2] ** 2 + a[:, 1:nrope:2] ** 2
    assert rel(pn(r), pn(v)) < 1e-14                                          # pair norms kept
    assert rel(O.rope_apply(r, pos, nrope, hd, 500000.0, inverse=True), v) < 1e-14
    assert np.array_equal(O.rope_apply(v, np.zeros(10, int), nrope, hd), v)   # pos 0 = identity
    # relative position: <R(p)q, R(k)k> depends only on p - k, per head
    q, k = v[0:1], v[1:2]
    for p1, p2, sh in ((5, 2, 100), (77, 1000, 3)):
        a = O.rope_apply(q, np.array([p1]), nrope, hd) * O.rope_apply(k, np.array([p2]), nrope, hd)
        b = O.rope_apply(q, np.array([p1 + sh]), nrope, hd) * O.rope_apply(k, np.array([p2 + sh]), nrope, hd)
        for h in range(nrope // hd):
            sl = slice(h * hd, (h + 1) * hd)
            assert abs(a[0, sl].sum() - b[0, sl].sum()) < 1e-11


def test_rope_is_complex_multiplication():
    # textbook reduction: rotating the pair (e, o) is multiplying e + i o by exp(i angle)
    rng = np.random.default_rng(13)
    hd, nrope = 8, 16
    v = rng.standard_normal((4, 24))
    pos = np.array([0, 1, 17, 4095])
    r = O.rope_apply(v, pos, nrope, hd, 500000.0)
    tv = torch.from_numpy(v[:, :nrope].copy()).reshape(4, nrope // 2, 2)
    cz = torch.view_as_complex(tv.contiguous())
    ang = torch.from_numpy(pos.astype(np.float64))[:, None] * torch.from_numpy(
        np.tile(O.rope_inv_freq(hd, 500000.0), nrope // hd))[None, :]
    rot = torch.view_as_real(cz * torch.polar(torch.ones_like(ang), ang)).reshape(4, nrope)
    assert rel(r[:, :nrope], rot.numpy()) < 1e-14


# ---------------------------------------------------------------- 8B-shaped block

def rand_8b(M=3, d=8, f=6, hd=4, nq=2, nkv=1, seed=14, wscale=0.3):
    rng = np.random.default_rng(seed)
    nqkv = (nq + 2 * nkv) * hd
    return dict(o=rng.standard_normal((M, d)), z=rng.standard_normal((M, d)),
                Wo=rng.standard_normal((d, d)) * wscale, W1=rng.standard_normal((d, 2 * f)) * wscale,
                W2=rng.standard_normal((f, d)) * wscale, gamma2=rng.uniform(0.5, 1.5, d),
                gamma1=rng.uniform(0.5, 1.5, d), Wqkv=rng.standard_normal((d, nqkv)) * wscale,
                dqkv=rng.standard_normal((M, nqkv)), dres=rng.standard_normal((M, d))), \
        (nq + nkv) * hd, hd


def _8b(inp, pos, nrope, hd, theta=500000.0):
    fw = O.block8b_fwd(inp["o"], inp["z"], inp["Wo"], inp["W1"], inp["W2"], inp["gamma2"],
                       inp["gamma1"], inp["Wqkv"], pos, nrope, hd, theta)
    return fw


def test_block8b_backward_finite_differences():
    inp, nrope, hd = rand_8b()
    pos = np.array([0, 3, 11])
    keys = ("o", "z", "Wo", "W1", "W2", "gamma2", "gamma1", "Wqkv")

    def L(vals):
        fw = _8b(vals, pos, nrope, hd)
        return float(np.sum(fw["qkv"] * inp["dqkv"]) + np.sum(fw["out"] * inp["dres"]))

    fw = _8b(inp, pos, nrope, hd)
    bw = O.block8b_bwd(fw, inp["o"], inp["Wo"], inp["W1"], inp["W2"], inp["gamma2"], inp["gamma1"],
                       inp["Wqkv"], inp["dqkv"], inp["dres"], pos, nrope, hd)
    gname = {"o": "do", "z": "dz", "Wo": "dWo", "W1": "dW1", "W2": "dW2", "gamma2": "dgamma2",
             "gamma1": "dgamma1", "Wqkv": "dWqkv"}
    for k in keys:
        fd = np.zeros_like(inp[k])
        for idx in np.ndindex(inp[k].shape):
            vals = {kk: np.array(inp[kk], copy=True) for kk in inp}
            vals[k][idx] += 1e-6
            lp = L(vals)
            vals[k][idx] -= 2e-6
            fd[idx] = (lp - L(vals)) / 2e-6
        assert rel(bw[gname[k]], fd) < 1e-6, k


def test_block8b_matches_torch_autograd():
    inp, nrope, hd = rand_8b(M=4, d=16, f=8, hd=4, nq=2, nkv=1, seed=15)
    pos = np.array([0, 1, 2, 3000])
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=k not in ("dqkv", "dres"))
         for k, v in inp.items()}
    h = t["o"] @ t["Wo"] + t["z"]
    h2 = F.rms_norm(h, (16,), t["gamma2"], 1e-6)
    y = h2 @ t["W1"]
    out = (F.silu(y[:, 0::2]) * y[:, 1::2]) @ t["W2"] + h
    q_in = F.rms_norm(out, (16,), t["gamma1"], 1e-6)
    pre = q_in @ t["Wqkv"]
    ang = torch.tensor(pos, dtype=torch.float64)[:, None] * torch.tensor(
        np.tile(O.rope_inv_freq(hd, 500000.0), nrope // hd))[None, :]
    cz = torch.view_as_complex(pre[:, :nrope].reshape(4, nrope // 2, 2).contiguous())
    rot = torch.view_as_real(cz * torch.polar(torch.ones_like(ang), ang)).reshape(4, nrope)
    qkv = torch.cat([rot, pre[:, nrope:]], 1)
    ((qkv * t["dqkv"]).sum() + (out * t["dres"]).sum()).backward()
    fw = _8b(inp, pos, nrope, hd)
    bw = O.block8b_bwd(fw, inp["o"], inp["Wo"], inp["W1"], inp["W2"], inp["gamma2"], inp["gamma1"],
                       inp["Wqkv"], inp["dqkv"], inp["dres"], pos, nrope, hd)
    assert rel(fw["qkv"], qkv.detach().numpy()) < 1e-13
    assert rel(fw["out"], out.detach().numpy()) < 1e-13
    for k, g in {"o": "do", "z": "dz", "Wo": "dWo", "W1": "dW1", "W2": "dW2", "gamma2": "dgamma2",
                 "gamma1": "dgamma1", "Wqkv": "dWqkv"}.items():
        assert rel(bw[g], t[k].grad.numpy()) < 1e-12, k


def test_block8b_qkv_statistic_through_rotation():
    # s' = (1/d) sumcols(dqkv_pre * qkv_pre) = (1/d) sumcols(dqkv * qkv): the
    # rotation preserves dot products pair by pair.
    inp, nrope, hd = rand_8b(M=5, d=8, f=6, seed=16)
    pos = np.array([0, 9, 100, 4095, 7])
    fw = _8b(inp, pos, nrope, hd)
    bw = O.block8b_bwd(fw, inp["o"], inp["Wo"], inp["W1"], inp["W2"], inp["gamma2"], inp["gamma1"],
                       inp["Wqkv"], inp["dqkv"], inp["dres"], pos, nrope, hd)
    a = np.sum(bw["dqkv_pre"] * fw["qkv_pre"], axis=1)
    b = np.sum(inp["dqkv"] * fw["qkv"], axis=1)
    assert rel(a, b) < 1e-13
    assert rel(bw["s1"], b / 8) < 1e-12


def test_block8b_reparam_equals_canonical():
    # delayed row scales through both RMSNorms, s and s1 from the relocated form
    inp, nrope, hd = rand_8b(M=5, d=16, f=12, hd=8, nq=2, nkv=1, seed=18)
    pos = np.array([0, 1, 5, 100, 4095])
    args = (inp["o"], inp["z"], inp["Wo"], inp["W1"], inp["W2"], inp["gamma2"], inp["gamma1"],
            inp["Wqkv"], pos, nrope, hd)
    fc = O.block8b_fwd(*args)
    fr = O.block8b_fwd_reparam(*args)
    for k in ("h", "r", "y", "a", "out", "r1", "qkv"):
        assert rel(fr[k], fc[k]) < 1e-12, k
    bargs = (inp["o"], inp["Wo"], inp["W1"], inp["W2"], inp["gamma2"], inp["gamma1"], inp["Wqkv"],
             inp["dqkv"], inp["dres"], pos, nrope, hd)
    bc = O.block8b_bwd(fc, *bargs)
    br = O.block8b_bwd_reparam(fr, *bargs)
    for k in ("s1", "s", "dout", "dz", "do", "dWo", "dW1", "dW2", "dWqkv", "dgamma1", "dgamma2"):
        assert rel(br[k], bc[k]) < 1e-11, k
    so = O.block8b_bwd_reparam(fr, *bargs, stat_only=True)
    assert rel(so["s"], bc["s"]) < 1e-11 and "dW1" not in so
    # storage mode rounds exactly the bf16-stored tensors
    frs = O.block8b_fwd_reparam(*args, store_bf16=True)
    for k in ("h", "hg", "a", "out", "outg", "qkv"):
        assert np.array_equal(frs[k], O.bf16_round(frs[k])), k
    assert rel(frs["qkv"], fc["qkv"]) < 2e-2


# ---------------------------------------------------------------- planted mistakes

def test_planted_mistakes_are_caught(monkeypatch):
    """Plants plausible mistakes in the oracle (CPU only) and checks that at
    least one pin above would catch each one."""
    inp = rand_block(M=2, d=8, f=8, seed=17)
    assert fd_block_error(inp) < 1e-6
    # 1) silu' replaced by sigmoid (dropped term)
    with monkeypatch.context() as mp:
        mp.setattr(O, "silu_grad", O.sigmoid)
        assert fd_block_error(inp) > 1e-3
    # 2) gate and up swapped in the forward only
    with monkeypatch.context() as mp:
        mp.setattr(O, "swiglu", lambda y: O.silu(y[:, 1::2]) * y[:, 0::2])
        assert fd_block_error(inp) > 1e-3
    # 3) eps outside the square root
    with monkeypatch.context() as mp:
        mp.setattr(O, "rms_factor", lambda h, eps=1e-6: 1.0 / (np.sqrt(np.mean(h * h, 1)) + eps))
        g = GOLD["block_example"]
        x = np.array([g["inputs"]["x"]], float)
        fw = O.mlp_fwd(x, np.array([g["inputs"]["z"]]), np.eye(2), np.eye(2),
                       np.array([[2.0, -1.0]]), np.array([1.0, 0.5]))
        assert abs(fw["r"][0] - g["r"]) > 1e-9


# ---------------------------------------------------------------- tensor-core GEMM model

U = 2.0 ** -23  # fp32 spacing just above 1


def test_tc_matmul_exact_when_nothing_rounds():
    # small integers: every group sum and every accumulator value is exact in fp32
    rng = np.random.default_rng(3)
    A = rng.integers(-8, 9, (5, 64)).astype(np.float64)
    B = rng.integers(-8, 9, (64, 7)).astype(np.float64)
    out = O.tc_matmul(A, B)
    assert out.dtype == np.float32
    assert np.array_equal(out.astype(np.float64), A @ B)


def test_tc_matmul_truncates_once_per_group_of_16():
    # row [1, 2^-25 x 31] times ones, K = 32. Group 1 sums exactly to
    # 1 + 15 * 2^-25 = 1 + 3.75 u and the accumulator keeps 1 + 3 u (toward
    # zero); group 2 adds 16 * 2^-25 = 4 u exactly: 1 + 7 u. Rounding to
    # nearest would give 1 + 8 u; truncating every product would give 1.
    a = np.full((1, 32), 2.0 ** -25)
    a[0, 0] = 1.0
    b = np.ones((32, 1))
    assert float(O.tc_matmul(a, b)[0, 0]) == 1.0 + 7 * U
    assert float(O.tc_matmul(-a, b)[0, 0]) == -(1.0 + 7 * U)  # toward zero on both sides
    # with one group of 32 the sum 1 + 7.75 u is truncated once: 1 + 7 u too,
    # while groups of 1 truncate every 2^-25 away
    assert float(O.tc_matmul(a, b, group=32)[0, 0]) == 1.0 + 7 * U
    assert float(O.tc_matmul(a, b, group=1)[0, 0]) == 1.0


def test_tc_matmul_error_is_within_the_truncation_bound_and_biased_to_zero():
    # K/16 truncating additions each lose less than one fp32 ulp of the
    # running sum, always toward zero
    rng = np.random.default_rng(4)
    A = O.bf16_round(rng.standard_normal((64, 2048)))
    B = O.bf16_round(rng.standard_normal((2048, 48)) * 0.02)
    exact = A @ B
    got = O.tc_matmul(A, B).astype(np.float64)
    # |partial sums| <= sum_k |a_k b_k|: a bound on every running value
    absmax = np.abs(A) @ np.abs(B)
    ulp = absmax * 2.0 ** -23
    assert np.all(np.abs(got - exact) <= (2048 / 16) * ulp)
    assert np.mean((got - exact) * np.sign(exact)) < 0  # biased toward zero
    assert rel(got, exact) > 10 * rel((A.astype(np.float32) @ B.astype(np.float32)), exact)


def test_fp32_mode_of_the_rewritten_block_is_fp32_and_close():
    # the fp32 mode runs the same steps; on a small block it agrees with the
    # fp64 mode to fp32-level error (nothing is stored in bf16 here)
    b = rand_block(M=4, d=32, f=32, seed=5)
    args = (b["x"], b["z"], b["W0"], b["W1"], b["W2"], b["gamma"])
    f64 = O.mlp_fwd_reparam(*args)
    f32 = O.mlp_fwd_reparam(*args, fp32=True)
    assert f32["out"].dtype == np.float32 and f32["r"].dtype == np.float32
    assert rel(f32["out"], f64["out"]) < 1e-5
    g64 = O.mlp_bwd_reparam(f64, b["x"], b["W0"], b["W1"], b["W2"], b["gamma"], b["dout"])
    g32 = O.mlp_bwd_reparam(f32, b["x"], b["W0"], b["W1"], b["W2"], b["gamma"], b["dout"], fp32=True)
    assert rel(g32["s"], g64["s"]) < 1e-4 and rel(g32["dx"], g64["dx"]) < 1e-5
