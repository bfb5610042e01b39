"""Write tests/golden/tile_counts.json from the CPU oracle only.

Per-round tile tables and modelled ring critical paths (sum over rounds of
the busiest device's tile count) for the benchmark workloads, all three
placements (striped, contiguous, zig-zag).  Small workloads use the oracle's pair-by-pair brute force; the
large ones its closed forms (which the oracle tests pin to the brute force).
Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

WORKLOADS = [
    # name, S, N, T
    ("tiny S=256 N=4 T=16", 256, 4, 16),
    ("tiny S=256 N=4 T=64", 256, 4, 64),
    ("short S=8192 N=8 T=128", 8192, 8, 128),
    ("mid S=65536 N=8 T=128", 65536, 8, 128),
    ("long S=262144 N=8 T=128", 262144, 8, 128),
    ("vlong S=786432 N=16 T=128", 786432, 16, 128),
]


def main():
    out = {"source": "oracle.tile_counts_bruteforce (S <= 8192) / oracle.tile_counts_closed",
           "counts_are": "per (batch, head); full/partial [round r][device d]",
           "workloads": []}
    for name, S, N, T in WORKLOADS:
        entry = {"name": name, "S": S, "N": N, "T": T}
        for lname, layout in (("striped", oracle.STRIPED), ("contiguous", oracle.CONTIGUOUS),
                              ("zigzag", oracle.ZIGZAG)):
            if S <= 8192:
                full, part = oracle.tile_counts_bruteforce(S, N, T, T, layout)
            else:
                full, part = oracle.tile_counts_closed(S, N, T, layout)
            entry[lname] = {"full": full.tolist(), "partial": part.tolist(),
                            "critical_path": oracle.critical_path(full, part),
                            "total": int(full.sum() + part.sum())}
        out["workloads"].append(entry)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tile_counts.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
