"""Writes the fp64 oracle's full forward of a linear cross-entropy configuration
to tests/golden: the mean loss over every valid token and the lse of every
token, for llama3 (8192 tokens x hidden 4096 x vocabulary 128256, seed 3) and
qwen32768 (the Qwen-7B head of the benchmark's chain, 32768 tokens x 4096 x
151936, seed 4); 10 % of the labels are ignored in both.  With every token's
lse stored, the tests can also form rows of dW exactly at these shapes.

The oracle computes the unchunked definition one row at a time (about 0.4 s a
row on one core), so the rows are split over worker processes (spawned, each
regenerating the seeded inputs).  Only datagen/ (the inputs) and oracle/ (the
arithmetic) are used.  Run from the repository root:

    python tests/golden/make_linear_ce_lse.py llama3|qwen32768 [workers]
"""
import json
import multiprocessing as mp
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
HERE = os.path.dirname(os.path.abspath(__file__))
CONFIGS = {
    # name: (workload call, H, V, seed, stride of the stored lse rows, output file)
    "llama3": ("linear_ce_llama3()", 4096, 128256, 3, 1, "linear_ce_llama3_lse.json"),
    "qwen32768": ("qwen_chain(32768)['linear_ce']", 4096, 151936, 4, 1, "linear_ce_qwen32768_lse.json"),
}


def _inputs(name):
    sys.path.insert(0, ROOT)
    from datagen import workloads
    c = eval("workloads." + CONFIGS[name][0], {"workloads": workloads})
    return c.make("X"), c.make("W"), c.make("labels")


def _rows(args):
    name, lo, hi = args
    sys.path.insert(0, ROOT)
    import oracle
    X, W, lab = _inputs(name)
    r = oracle.linear_ce_rows_fwd(X, W, lab, np.arange(lo, hi))
    return lo, r["lse"].tolist(), r["loss_term"].tolist()


def main():
    name = sys.argv[1]
    workers = int(sys.argv[2]) if len(sys.argv) > 2 else os.cpu_count()
    call, H, V, seed, stride, out = CONFIGS[name]
    lab = _inputs(name)[2]
    T = lab.shape[0]
    jobs = [(name, lo, min(T, lo + 64)) for lo in range(0, T, 64)]
    lse = [0.0] * T
    term = [0.0] * T
    t0 = time.time()
    with mp.get_context("spawn").Pool(workers) as pool:
        for lo, l, lt in pool.imap_unordered(_rows, jobs):
            lse[lo:lo + len(l)] = l
            term[lo:lo + len(lt)] = lt
    valid = lab != -100
    n_valid = int(valid.sum())
    loss = float(np.sum(np.array(term)[valid]) / n_valid)
    doc = {
        "source": f"fp64 oracle (oracle.linear_ce_rows_fwd, the unchunked definition) on datagen.workloads.{call}; "
                  "written by tests/golden/make_linear_ce_lse.py",
        "T": int(T), "H": H, "V": V, "seed": seed, "ignore_index": -100, "n_valid": n_valid,
        "loss_mean": loss, "lse_row_stride": stride, "lse": lse[::stride],
    }
    with open(os.path.join(HERE, out), "w") as f:
        json.dump(doc, f)
    print(f"wrote {out}: loss {loss:.10f}, {T} rows, {time.time() - t0:.0f} s with {workers} workers")


if __name__ == "__main__":
    main()
