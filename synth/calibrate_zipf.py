"""Pick the Zipf bias scale c of the skewed prefill workload with the oracle's
router: the largest per-expert load should be about ten times the mean.

Prints the realised load statistics of every workload's routing as well.
Run: python synth/calibrate_zipf.py [c ...]
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import oracle  # noqa: E402
import synth  # noqa: E402


def loads(w, c=None):
    w = dict(w)
    if c is not None:
        synth.ZIPF_C = c
    x = synth.x_rows(w, np.arange(w["T"]))
    logits, _ = oracle.router_logits(x, synth.router_weight(w))
    idx, _, _ = oracle.router_select(logits, synth.router_bias(w), w["k"])
    cnt = np.bincount(idx.ravel(), minlength=w["E"])
    return cnt


def main():
    cs = [float(a) for a in sys.argv[1:]]
    for name, w in synth.WORKLOADS.items():
        if name == "prefill16384_mxfp8_zipf" and cs:
            for c in cs:
                cnt = loads(w, c)
                print(f"{name} c={c}: max/mean={cnt.max() / cnt.mean():.2f} empty={int((cnt == 0).sum())}")
            continue
        cnt = loads(w)
        print(f"{name}: touched={int((cnt > 0).sum())} max={cnt.max()} mean={cnt.mean():.2f} "
              f"max/mean={cnt.max() / cnt.mean():.2f} empty={int((cnt == 0).sum())}")


if __name__ == "__main__":
    main()
