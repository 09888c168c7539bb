"""Writes closed_forms.json: values fixed by mathematics alone, worked by hand
and evaluated here with mpmath at 40 significant digits. It imports nothing
from the oracle or from the CUDA library.

Citations (page title, section):
  * ln V for all-zero logits: "Reading notes on CODA", s2 "Cross-entropy loss"
    (l_i = -h_{i,y_i} + log sum_k exp h_{i,k}; with every logit 0 it is log V);
    the same definition on eight bf16-exact logits (ce_exact8).
  * RoPE frequencies and rotations: "CODA: Rewriting Transformer Blocks as
    GEMM-Epilogue Programs" (pith.science), Fig. 7 caption (RoPE rotates each
    feature pair); theta = 500000 and head dim 128 are the Llama-3-8B-shaped
    workload's settings.
  * SiLU values: the SwiGLU gate activation, same Fig. 7 caption.
  * The worked block example: "Reading notes on CODA", s2
    "GEMM -> Residual -> RMSNorm -> GEMM" and s3 "Reverse Fusion".

Run:  python tests/golden/make_closed_forms.py
"""
import json
import os

import mpmath as mp

mp.mp.dps = 40


def f(v):
    return float(mp.nstr(v, 30))


def main():
    out = {}

    # LM head with W = 0: every logit is 0, so LSE = loss = ln V.
    out["ln_V_128256"] = f(mp.log(128256))

    # Four logits [0, ln2, ln3, 0]: sum of exps = 1 + 2 + 3 + 1 = 7.
    out["ce_small"] = {"logits": ["0", "ln2", "ln3", "0"], "lse": f(mp.log(7)),
                       "loss_target2": f(mp.log(mp.mpf(7) / 3)),
                       "loss_target0": f(mp.log(7))}

    # Eight logits that bf16 holds exactly: lse = ln sum exp, loss_t = lse - l_t.
    lg = ["0", "1", "2", "0.5", "-1", "3", "0", "0.25"]
    lse8 = mp.log(sum(mp.exp(mp.mpf(v)) for v in lg))
    out["ce_exact8"] = {"logits": [float(v) for v in lg], "lse": f(lse8),
                        "loss": [f(lse8 - mp.mpf(v)) for v in lg]}

    # RoPE inverse frequencies theta^(-2i/128), theta = 5e5.
    th = mp.mpf(500000)
    out["rope_inv_freq_5e5_128"] = {str(i): f(mp.power(th, -mp.mpf(2 * i) / 128))
                                    for i in (0, 1, 2, 31, 63)}
    # head_dim 4, theta 1e4: theta_0 = 1, theta_1 = 0.01. v = [1, 0, 0, 1] at pos 3:
    # pair 0 -> (cos 3, sin 3), pair 1 = (0, 1) rotated by 0.03 -> (-sin .03, cos .03).
    out["rope_hd4_pos3"] = [f(mp.cos(3)), f(mp.sin(3)), f(-mp.sin(mp.mpf("0.03"))),
                            f(mp.cos(mp.mpf("0.03")))]

    # SiLU and its derivative.
    sig = lambda t: 1 / (1 + mp.exp(-t))
    silu = lambda t: t * sig(t)
    dsilu = lambda t: sig(t) * (1 + t * (1 - sig(t)))
    out["silu"] = {"1": f(silu(1)), "-1": f(silu(-1)), "3": f(silu(3))}
    out["dsilu"] = {"0": f(dsilu(0)), "1": f(dsilu(1)), "-2": f(dsilu(-2))}

    # Worked block example, M = 1, d = 2, f = 1, eps = 1e-6:
    #   x = [1, 2], z = [0.5, -1], W0 = I  ->  h = [1.5, 1.0]
    #   mean h^2 = (2.25 + 1)/2 = 1.625  ->  r = 1/sqrt(1.625 + 1e-6)
    #   gamma = [1, 0.5]  ->  h2 = r [1.5, 0.5]
    #   W1 = I (2x2, column 0 = gate, column 1 = up)  ->  g = 1.5 r, u = 0.5 r
    #   a = silu(g) u ;  W2 = [[2, -1]]  ->  out = [2a, -a]
    # Backward for dout = [1, 1]:
    #   da = 2 - 1 = 1 ; dg = u silu'(g) ; du = silu(g)
    #   dh2 = dy (W1 = I) ; n = r h ; dgamma = dh2 * n ; dn = gamma * dh2
    #   s = (dn . n)/2 ; dh = r (dn - s n) ; dx = dh ; dW0 = x^T dh
    #   dW1 = h2^T dy ; dW2 = [a, a]
    eps = mp.mpf("1e-6")
    x = [mp.mpf(1), mp.mpf(2)]
    z = [mp.mpf("0.5"), mp.mpf(-1)]
    gam = [mp.mpf(1), mp.mpf("0.5")]
    h = [x[0] + z[0], x[1] + z[1]]
    r = 1 / mp.sqrt((h[0] ** 2 + h[1] ** 2) / 2 + eps)
    n = [r * h[0], r * h[1]]
    h2 = [n[0] * gam[0], n[1] * gam[1]]
    g, u = h2[0], h2[1]
    a = silu(g) * u
    outv = [2 * a, -a]
    da = mp.mpf(1)
    dg = da * u * dsilu(g)
    du = da * silu(g)
    dy = [dg, du]
    dh2 = dy
    dgamma = [dh2[0] * n[0], dh2[1] * n[1]]
    dn = [gam[0] * dh2[0], gam[1] * dh2[1]]
    s = (dn[0] * n[0] + dn[1] * n[1]) / 2
    dh = [r * (dn[0] - s * n[0]), r * (dn[1] - s * n[1])]
    dW0 = [[x[0] * dh[0], x[0] * dh[1]], [x[1] * dh[0], x[1] * dh[1]]]
    dW1 = [[h2[0] * dy[0], h2[0] * dy[1]], [h2[1] * dy[0], h2[1] * dy[1]]]
    out["block_example"] = {
        "inputs": {"x": [1, 2], "z": [0.5, -1], "W0": [[1, 0], [0, 1]],
                   "W1": [[1, 0], [0, 1]], "W2": [[2, -1]], "gamma": [1, 0.5],
                   "dout": [1, 1], "eps": 1e-6},
        "h": [f(v) for v in h], "r": f(r), "y": [f(g), f(u)], "a": f(a),
        "out": [f(v) for v in outv], "s": f(s), "dh": [f(v) for v in dh],
        "dgamma": [f(v) for v in dgamma], "dW0": [[f(v) for v in row] for row in dW0],
        "dW1": [[f(v) for v in row] for row in dW1], "dW2": [[f(a)], [f(a)]],
        "dy": [f(v) for v in dy],
    }

    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_forms.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1, sort_keys=True)
        fh.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
