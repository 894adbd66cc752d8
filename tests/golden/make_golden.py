"""Writes tests/golden/tiny_fp32_oracle_rows.txt from the oracle alone.

The pages print no worked MLA example, so this fixture is a regression anchor, not
a published value: the oracle's output for a few rows of the tiny fp32 workload
(seed 0 synthetic inputs).  It calls only ``oracle`` and the seeded input generator.
Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from head_latent_attention_rmsnorm_gb300 import configs, inputs  # noqa: E402

ROWS = (0, 1, 63, 64, 127)


def main():
    cfg = configs.TINY
    inp = {k: v.double().numpy() for k, v in inputs.prefill_inputs(cfg, seed=0).items()}
    out, lse = oracle.mla_explicit(**inp, n_heads=cfg.n_heads, q_offset=0, causal=True,
                                   base=cfg.rope_base, eps=cfg.rms_eps)
    path = os.path.join(ROOT, "tests", "golden", "tiny_fp32_oracle_rows.txt")
    with open(path, "w") as f:
        f.write("# tiny fp32 MLA prefill (B=1,S=128,H=4,Dk=64,Dn=32,Dr=16,Dv=32), seed 0, causal\n")
        f.write("# written by tests/golden/make_golden.py from the oracle; columns:\n")
        f.write("# row head lse out[0..7]\n")
        for i in ROWS:
            for h in range(cfg.n_heads):
                vals = " ".join("%.17g" % v for v in out[0, i, h, :8])
                f.write("%d %d %.17g %s\n" % (i, h, lse[0, h, i], vals))


if __name__ == "__main__":
    main()
