"""Write tests/golden/tiny_layer.npz: the oracle's output on the tiny workload.

No page prints a worked numeric example, so this file is not a page value: it
is written by this script, which calls only ``oracle/`` and ``synthetic/``.
It guards against the oracle changing (or differing between the x86 host and
the Arm GPU host) without notice. Re-run only when a change to the oracle's
arithmetic is justified by a passage of the pages, and say which one.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle      # noqa: E402
import synthetic   # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_layer.npz")


def compute():
    wl = synthetic.WORKLOADS["tiny"]
    x = synthetic.activations(wl.seed, wl.T, wl.H)
    Wr = synthetic.router_weights(wl.seed, 0, wl.E, wl.H)
    ws = synthetic.shared_gate_weights(wl.seed, 0, wl.H)
    r = oracle.layer(wl, 0, x, Wr, ws, want_probs=True)
    return dict(x=x, ids=r["ids"], w=r["w"], gate=r["gate"], out64=r["out64"],
                out_bf16=r["out_bf16"], probs=r["probs"])


if __name__ == "__main__":
    np.savez(OUT, **compute())
    print(OUT)
