"""Approximation error of the library's FAVOR+ output against exact softmax
attention as the number of random features m grows: the shape of Fig. 4 of
Rethinking Attention with Performers (§4.2) -- L = 4096, d = 16, m swept,
15 samples, orthogonal (ORF) against iid projections.

Inputs as the approximation-error workload states them: B = 1, H = 8,
L = 4096, d = dv = 16, Q, K, V ~ N(0, 1) scaled by d^-1/4, fp32, data scale 1.
Sample `seed` draws Q, K, V from Generator(PCG64(seed)) once (the same
inputs for every m) and omega from Generator(PCG64(seed + 1000)) per (m,
ORF/iid).  For every point the table gives

  * the MSE of the library's output against exact softmax attention (the
    oracle's softmax_attention, float64), mean and std over the samples;
  * the largest element-wise error (1%-of-row floor) of the library's output
    against the FAVOR+ oracle on the same omega -- the parity check at that
    point.

Run where the library is built and a GPU is present:

    python tests/approx_report.py [--seeds 15] [--out profiles/approx_error_fig4.md]
"""
from __future__ import annotations

import argparse
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle as O  # noqa: E402
from synth import CONFIGS, make_omega_iid, make_omega_orf, make_qkv  # noqa: E402

MS = (16, 32, 64, 128, 256)


def sample_inputs(seed: int):
    w = CONFIGS["approx_f32"]
    rng = np.random.Generator(np.random.PCG64(seed))
    q, k, v = make_qkv(rng, w.B, w.H, w.L, w.d, w.dv, w.std)
    sc = np.float32(w.input_scale)
    return w, q * sc, k * sc, v * sc


def sample_omega(seed: int, m: int, ortho: bool, H: int, d: int):
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    make = make_omega_orf if ortho else make_omega_iid
    return np.stack([make(rng, m, d) for _ in range(H)]).astype(np.float32)


def curve(seeds=range(15), ms=MS):
    """{(m, 'orf'|'iid'): {'mse': [...per seed], 'parity': max error}} from the library."""
    import torch

    import random_feature_gb300 as R

    res = {}
    for seed in seeds:
        w, q, k, v = sample_inputs(seed)
        exact = O.softmax_attention(q, k, v, w.data_scale)
        qd, kd, vd = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (q, k, v))
        for m in ms:
            for ortho in (True, False):
                om = sample_omega(seed, m, ortho, w.H, w.d)
                with R.Favor(w.H, m, w.d, w.dv, "softmax_pos", "f32", om, w.data_scale, w.B, w.L) as f:
                    got = f.attn(qd, kd, vd).double().cpu().numpy()
                ref = O.favor_bidir(q, k, v, om, w.data_scale)
                ent = res.setdefault((m, "orf" if ortho else "iid"), {"mse": [], "parity": 0.0})
                ent["mse"].append(float(np.mean((got - exact) ** 2)))
                ent["parity"] = max(ent["parity"], O.elem_rel_err(got, ref))
    return res


def table(res, nseeds: int, seconds: float) -> str:
    ms = sorted({m for m, _ in res})
    lines = [
        "# Approximation error vs m (Fig. 4 shape): the library's FAVOR+ output against exact softmax",
        "",
        "Workload: B=1, H=8, L=4096, d=dv=16, Q, K, V ~ N(0,1) * 16^-1/4 (fp32), data scale 1, "
        f"positive features; {nseeds} samples (seeds 0..{nseeds - 1}): inputs from PCG64(seed), "
        "omega from PCG64(seed + 1000) per (m, ORF/iid).",
        "",
        "Command: `python tests/approx_report.py` (GPU; library built in-tree); "
        f"{seconds:.0f} s including the float64 oracle.",
        "",
        "| m | ORF MSE mean | ORF MSE std | iid MSE mean | iid MSE std | ORF / iid | parity (ORF, iid) |",
        "|---|---|---|---|---|---|---|",
    ]
    for m in ms:
        o, i = res[(m, "orf")], res[(m, "iid")]
        om_, os_ = np.mean(o["mse"]), np.std(o["mse"])
        im_, is_ = np.mean(i["mse"]), np.std(i["mse"])
        lines.append(f"| {m} | {om_:.4e} | {os_:.2e} | {im_:.4e} | {is_:.2e} | {om_ / im_:.3f} | "
                     f"{o['parity']:.1e}, {i['parity']:.1e} |")
    lines += ["",
              "MSE: mean over heads, queries and value columns of (library - exact softmax)^2 per sample, then "
              "mean and std over samples.  Parity: largest element-wise error (1%-of-row floor) of the library "
              "against the float64 FAVOR+ oracle on the same omega over all samples (the fp32 bar is 1e-4)."]
    return "\n".join(lines) + "\n"


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--seeds", type=int, default=15)
    ap.add_argument("--out", default=os.path.join(ROOT, "profiles", "approx_error_fig4.md"))
    a = ap.parse_args()
    t0 = time.time()
    res = curve(range(a.seeds))
    text = table(res, a.seeds, time.time() - t0)
    with open(a.out, "w") as f:
        f.write(text)
    print(text)


if __name__ == "__main__":
    main()
