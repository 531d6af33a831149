"""One worker of the all-core CPU timing of the oracle's paged decode.

The parent (bench.py's CPU baseline) writes a sample of a decode workload
(the compacted K/V pool of its sequences as bf16 bit patterns, the block
tables, context lengths and queries) to a directory and starts one worker
per host core, each a separate process, so that the oracle's NumPy work runs
on every core at once.  A worker maps the arrays, reads its share of the
sequences once so its pages are resident, runs the oracle once on a short
context (NumPy's and BLAS's first-call set-up), prints "ready", waits for a
line on standard input, decodes its sequences `reps` times with the oracle
and prints the elapsed seconds as JSON.

    python tests/_oracle_pool.py <dir> <worker index>
"""
import json
import os
import sys
import time

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_v] = "1"

import numpy as np  # noqa: E402

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import attention as A  # noqa: E402


def main():
    d, w = sys.argv[1], int(sys.argv[2])
    meta = json.load(open(os.path.join(d, "meta.json")))
    load = lambda name: np.load(os.path.join(d, name + ".npy"), mmap_mode="r")
    k, v, tab, lens, q = load("k"), load("v"), load("tab"), load("lens"), load("q")
    mine = np.array(meta["assign"][w], dtype=np.int64)
    B = int(meta["block_size"])
    used = set()
    for s in mine:
        used.update(int(b) for b in tab[s, :-(-int(lens[s]) // B)])
    touch = 0
    for b in sorted(used):
        touch += int(k[b].view(np.uint16)[..., 0].sum()) + int(v[b].view(np.uint16)[..., 0].sum())
    if len(mine):
        # first calls into NumPy and BLAS carry one-time set-up: pay it on one
        # short context before the clock starts
        s0 = mine[:1]
        A.paged_decode(np.asarray(q[s0]), k, v, np.asarray(tab[s0]), np.minimum(np.asarray(lens[s0]), B),
                       float(meta["scale"]), B)
    print("ready", flush=True)
    sys.stdin.readline()
    t0 = time.perf_counter()
    for _ in range(int(meta["reps"])):
        if len(mine):
            A.paged_decode(np.asarray(q[mine]), k, v, np.asarray(tab[mine]), np.asarray(lens[mine]),
                           float(meta["scale"]), B)
    print(json.dumps({"elapsed": time.perf_counter() - t0, "touched": touch % 7}), flush=True)


if __name__ == "__main__":
    main()
