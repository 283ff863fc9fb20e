"""Triton's Philox-4x32 (tl.philox, 10 rounds), run in Triton's CPU interpreter.

Helper of tests/test_oracle_dropout.py, run as a child process with
TRITON_INTERPRET=1 (the interpreter must be on when triton is imported and when
its kernels run). Reads {"ctr": [[c0, c1, c2, c3], ...], "seed": [s, ...]} as
JSON on stdin and writes {"out": [[w0, w1, w2, w3], ...]}: row i is Philox of
counter ctr[i] under the key (seed[i] & 0xffffffff, seed[i] >> 32).
"""
import json
import sys

import numpy as np
import torch
import triton
import triton.language as tl


@triton.jit
def _philox_kernel(c_ptr, o_ptr, seed):
    c0 = tl.load(c_ptr)
    c1 = tl.load(c_ptr + 1)
    c2 = tl.load(c_ptr + 2)
    c3 = tl.load(c_ptr + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3, 10)
    tl.store(o_ptr, a)
    tl.store(o_ptr + 1, b)
    tl.store(o_ptr + 2, c)
    tl.store(o_ptr + 3, d)


def main():
    req = json.load(sys.stdin)
    out = []
    for ctr, seed in zip(req["ctr"], req["seed"]):
        c = torch.from_numpy(np.asarray(ctr, dtype=np.int64)).to(torch.uint32)
        o = torch.zeros(4, dtype=torch.uint32)
        _philox_kernel[(1,)](c, o, int(seed))  # one key per launch: the seed is a scalar argument
        out.append([int(x) for x in o.to(torch.int64).tolist()])
    json.dump({"out": out}, sys.stdout)


if __name__ == "__main__":
    main()
