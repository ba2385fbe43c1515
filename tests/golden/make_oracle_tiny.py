"""Writes oracle_tiny.txt: the oracle's logits for a tiny seeded model at its
first positions (greedy, from token 1). Calls only the seeded generator and the
oracle; rerun it only with a commit that says which reading of the pages
changed the oracle's arithmetic."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

CFG = dict(dim=16, hidden_dim=40, n_layers=2, n_heads=4, n_kv_heads=2, vocab_size=32,
           seq_len=8, rope_theta=10000.0, norm_eps=1e-5, shared_classifier=0, max_batch=1)
SEED, STD, POSITIONS = 7, 0.3, 4


def compute():
    blob = synth.make_blob(CFG, SEED, std=STD)
    m = oracle.Model(CFG, blob)
    tok, rows = 1, []
    for p in range(POSITIONS):
        lg = m.forward(tok, p)
        rows.append(np.asarray(lg, np.float64))
        tok = int(np.argmax(lg))
    m.close()
    return np.stack(rows)


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.txt")
    with open(out, "w") as f:
        f.write("# oracle logits, tiny model (see make_oracle_tiny.py): one position per line\n")
        for row in compute():
            f.write(" ".join(f"{v:.9e}" for v in row) + "\n")
    print(out)
