"""Write tiny_t64_d32.npz: the oracle's outputs for the 64-token, dk = dv = 32 workload.

Calls only the oracle (and the seeded input generator).  Rerun after a change to the
oracle's arithmetic that a passage of the pages justifies, and say which in the commit.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from hybrid_linear_attention_prefill_gb300.inputs import workload  # noqa: E402

if __name__ == "__main__":
    out, fin = oracle.prefill_inputs(workload("tiny_t64_d32"))
    np.savez_compressed(os.path.join(HERE, "tiny_t64_d32.npz"), out=out, final_state=fin)
    print("wrote", os.path.join(HERE, "tiny_t64_d32.npz"), out.shape, fin.shape)
