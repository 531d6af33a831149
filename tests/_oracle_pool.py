"""One worker of the all-core CPU timing of the oracle's paged decode or
prefill.

The parent (bench.py's CPU baseline) writes a sample of a workload to a
directory and starts one worker per host core, each a separate process, so
that the oracle's NumPy work runs on every core at once.  Decode: the
compacted K/V pool of the sample's sequences as bf16 bit patterns, the block
tables, context lengths and queries; each worker decodes its share of the
sequences.  Prefill (meta "mode": "prefill"): one sequence's K/V blocks, its
table and the last rows of its new positions; each worker computes its
share of those rows as one chunk at their positions.  A worker maps the
arrays, reads its blocks once so their pages are resident, runs the oracle
once on a short context (NumPy's and BLAS's first-call set-up), prints
"ready", waits for a line on standard input, runs its share `reps` times
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


def prefill_worker(d, w, meta, load):
    k, v, tab, q = load("k"), load("v"), load("tab"), load("q")
    a, b = meta["assign"][w]                          # rows [a, b) of the sampled rows
    B, end0 = int(meta["block_size"]), int(meta["first_pos"])
    touch = int(k.view(np.uint16)[..., 0].sum()) + int(v.view(np.uint16)[..., 0].sum())

    def run(lo, hi):
        # rows lo .. hi-1 sit at positions end0 + lo .. end0 + hi - 1: a chunk
        # of hi - lo new positions whose context ends at end0 + hi
        A.paged_prefill(np.asarray(q[lo:hi]), k, v, np.asarray(tab), np.array([0, hi - lo], dtype=np.int32),
                        np.array([end0 + hi], dtype=np.int32), float(meta["scale"]), B)

    if b > a:
        run(a, a + 1)
    print("ready", flush=True)
    sys.stdin.readline()
    t0 = time.perf_counter()
    for _ in range(int(meta["reps"])):
        if b > a:
            run(a, b)
    print(json.dumps({"elapsed": time.perf_counter() - t0, "touched": touch % 7}), flush=True)


def main():
    d, w = sys.argv[1], int(sys.argv[2])
    meta = json.load(open(os.path.join(d, "meta.json")))
    load = lambda name: np.load(os.path.join(d, name + ".npy"), mmap_mode="r")
    if meta.get("mode") == "prefill":
        prefill_worker(d, w, meta, load)
        return
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
