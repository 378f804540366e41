"""Write the oracle's single-linear-layer trajectory (64->32+bias, batch 128, 10 steps).

Calls only the oracle and the seeded input module.  The pages print no worked
example, so this file is a regression record of the oracle, not a pin of it:
the pins are the closed forms and brute-force checks in tests/test_oracle.py.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle as O      # noqa: E402
import workloads as W   # noqa: E402


def main():
    cfg = W.get_config("c1")
    hp = cfg.hp
    orc = O.KfacOracle(hp.ema_decay, hp.damping, hp.lr, hp.momentum, hp.weight_decay,
                       cfg.invert_every)
    kl, dl = cfg.layers
    w0, b0 = W.initial_params(cfg, 0)
    sk = O.LayerState("kron", kl.d_out, kl.d_in, kl.has_bias, w0, b0)
    sd = O.LayerState("diag", dl.d_out, dl.d_in, dl.has_bias, w0, b0)
    Wk, Wd = [], []
    for t in range(1, cfg.steps + 1):
        x = W.layer_inputs(cfg, 0, t)
        orc.step_kron(sk, x["a"], x["g"], x["grad_w"], x["grad_b"])
        orc.step_diag(sd, O.diag_factor(x["g"]), O.diag_factor(x["a"], 1), x["grad_w"], x["grad_b"])
        Wk.append(sk.W.copy())
        Wd.append(sd.W.copy())
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c1_oracle_trajectory.npz")
    np.savez_compressed(out, W=np.array(Wk), A=sk.A, G=sk.G, Wdiag=np.array(Wd))
    print("wrote", out)


if __name__ == "__main__":
    main()
