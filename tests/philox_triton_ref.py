"""Philox4x32-10 words from Triton's own implementation, for pinning the oracle.

Run as a child process with TRITON_INTERPRET=1 (Triton's CPU interpreter), so
no GPU is needed.  Reads {"ctrs": [[c0,c1,c2,c3], ...], "seeds": [...]} as
JSON on stdin and prints one JSON line: for every seed, for every counter,
the four output words.  Triton keys Philox with (lo32(seed), hi32(seed)).
"""
import json
import os
import sys

os.environ.setdefault("TRITON_INTERPRET", "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _philox_kernel(out_ptr, c_ptr, seed, n, BLOCK: tl.constexpr):
    offs = tl.arange(0, BLOCK)
    m = offs < n
    c0 = tl.load(c_ptr + offs * 4 + 0, mask=m, other=0).to(tl.uint32, bitcast=True)
    c1 = tl.load(c_ptr + offs * 4 + 1, mask=m, other=0).to(tl.uint32, bitcast=True)
    c2 = tl.load(c_ptr + offs * 4 + 2, mask=m, other=0).to(tl.uint32, bitcast=True)
    c3 = tl.load(c_ptr + offs * 4 + 3, mask=m, other=0).to(tl.uint32, bitcast=True)
    r0, r1, r2, r3 = tl.philox(seed, c0, c1, c2, c3, 10)
    tl.store(out_ptr + offs * 4 + 0, r0.to(tl.int32, bitcast=True), mask=m)
    tl.store(out_ptr + offs * 4 + 1, r1.to(tl.int32, bitcast=True), mask=m)
    tl.store(out_ptr + offs * 4 + 2, r2.to(tl.int32, bitcast=True), mask=m)
    tl.store(out_ptr + offs * 4 + 3, r3.to(tl.int32, bitcast=True), mask=m)


def main():
    req = json.loads(sys.stdin.read())
    ctrs = np.array(req["ctrs"], dtype=np.uint64).astype(np.uint32)
    n = ctrs.shape[0]
    block = 1 << max(0, (n - 1).bit_length())
    c = torch.from_numpy(ctrs.view(np.int32).reshape(-1).copy())
    result = []
    for seed in req["seeds"]:
        out = torch.zeros(n * 4, dtype=torch.int32)
        _philox_kernel[(1,)](out, c, int(seed), n, BLOCK=block)
        words = (out.numpy().view(np.uint32)).reshape(n, 4)
        result.append(words.astype(np.int64).tolist())
    print(json.dumps(result))


if __name__ == "__main__":
    main()
