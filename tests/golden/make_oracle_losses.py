"""Write the oracle's loss curve for a training workload to a JSON fixture.

Calls only the CPU oracle and the seeded input generators.  For the bf16 workloads the
stored curve is the fp32 oracle's: the loss of each of the first ``n`` steps (the
forward before that step's AdamW update) and the loss of one more forward after the
n-th update.  For an fp8 workload the oracle runs in its fp8 mode (e4m3 qkv and fc
products).  Usage:

    python tests/golden/make_oracle_losses.py gpt2_124m_bf16_b16_t1024 10
"""
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import gpt2_oracle as O                      # noqa: E402
from step_gpt_train_03_b300 import synth                 # noqa: E402


def main(name, n):
    w = synth.WORKLOADS[name]
    o = O.from_shape(w.shape, np.float32)
    o.keep_preatt = False
    o.fp8 = w.precision == "fp8"
    o.load(synth.init_params(w.shape, w.seed))
    batches = synth.workload_batches(w, n + 1)
    losses, secs = [], []
    for i in range(n):
        t0 = time.time()
        losses.append(o.step(*batches[i], w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, i + 1))
        secs.append(time.time() - t0)
        print(f"step {i}: loss {losses[-1]:.6f} ({secs[-1]:.1f} s)", flush=True)
    final = o.forward(*batches[n])
    print(f"after {n} updates: loss {final:.6f}", flush=True)
    out = {
        "workload": name, "oracle_dtype": "float32", "oracle_fp8": o.fp8, "steps": n,
        "losses": losses, "loss_after_updates": final,
        "note": "written by tests/golden/make_oracle_losses.py from the CPU oracle only",
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), f"{name}_oracle_losses.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main(sys.argv[1], int(sys.argv[2]))
