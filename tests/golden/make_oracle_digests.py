#!/usr/bin/env python
"""Writes the stored oracle digests of a full-size workload.

Runs the CPU oracle (and nothing else: inputs come from the seeded workload
generator) over every seed of a workload, in chunks of CHUNK seeds, and stores
per chunk the digest of its results (tests/digest.py) and its live-cell count,
keyed by the hash of the generated inputs.  The GPU parity test then compares
every extension of the batch against these digests.

  python tests/golden/make_oracle_digests.py --config 3 [--threads N]

The run can take hours on a few cores; it is resumable: chunks already in the
output file are kept, and the file is rewritten after every chunk.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gapped_smith_waterman_gb300 import workloads as W  # noqa: E402
from tests import digest as D  # noqa: E402

CHUNK = 4096


def out_path(config: int) -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), f"oracle_digest_cfg{config}.json")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--threads", type=int, default=os.cpu_count() or 1)
    ap.add_argument("--max-chunks", type=int, default=0, help="stop after this many new chunks (0: all)")
    args = ap.parse_args()
    w = W.make(args.config)
    ih = D.input_sha256(w)
    n = len(w.seeds)
    nch = (n + CHUNK - 1) // CHUNK
    path = out_path(args.config)
    doc = None
    if os.path.exists(path):
        doc = json.load(open(path))
        if doc.get("input_sha256") != ih or doc.get("chunk_seeds") != CHUNK:
            sys.exit(f"{path} holds digests of other inputs; move it away first")
    if doc is None:
        doc = {"workload": w.name, "config": args.config, "input_sha256": ih, "n_seeds": n,
               "chunk_seeds": CHUNK, "generated_by": "tests/golden/make_oracle_digests.py (CPU oracle only)",
               "chunks": [None] * nch, "live_cells": [None] * nch}
    done_new = 0
    for c in range(nch):
        if doc["chunks"][c] is not None:
            continue
        idx = np.arange(c * CHUNK, min(n, (c + 1) * CHUNK))
        t0 = time.time()
        ores, ocig, ooff = oracle.extend_batch(w, seeds=w.seeds[idx], nthreads=args.threads)
        doc["chunks"][c] = D.chunk_digest(*D.oracle_chunk(ores, ocig, ooff))
        doc["live_cells"][c] = int(ores["live_cells"].sum())
        tmp = path + ".tmp"
        with open(tmp, "w") as f:
            json.dump(doc, f, indent=0)
        os.replace(tmp, path)
        done_new += 1
        left = sum(x is None for x in doc["chunks"])
        print(f"chunk {c}: {time.time() - t0:.1f} s, {left} left", flush=True)
        if args.max_chunks and done_new >= args.max_chunks:
            break


if __name__ == "__main__":
    main()
