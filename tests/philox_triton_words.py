"""Philox4x32-10 output words from Triton's own generator, run on the CPU by
Triton's interpreter: an implementation of the generator independent of the
oracle's.  ``tl.randint4x(seed, offset)`` takes the counter (offset low word,
offset high word, 0, 0) and the key (seed low word, seed high word), the same
counter/key layout the dropout contract uses.

Usage: python philox_triton_words.py '<json: {"seeds": [...], "offsets": [...]}>'
Prints a JSON list, per seed, of per-offset lists of the four words.
"""
import json
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _words(out, seed, offs_ptr, N: tl.constexpr):
    i = tl.arange(0, N)
    a, b, c, d = tl.randint4x(seed, tl.load(offs_ptr + i))
    tl.store(out + i * 4 + 0, a)
    tl.store(out + i * 4 + 1, b)
    tl.store(out + i * 4 + 2, c)
    tl.store(out + i * 4 + 3, d)


def main():
    req = json.loads(sys.argv[1])
    offsets = [int(x) for x in req["offsets"]]
    n = 1 << max(0, (len(offsets) - 1).bit_length())
    offs = torch.tensor([o - (1 << 64) if o >= (1 << 63) else o for o in offsets] + [0] * (n - len(offsets)),
                        dtype=torch.int64)
    result = []
    for seed in req["seeds"]:
        seed = int(seed)
        out = torch.zeros(4 * n, dtype=torch.int32)
        _words[(1,)](out, seed - (1 << 64) if seed >= (1 << 63) else seed, offs, N=n)
        w = [x & 0xFFFFFFFF for x in out.tolist()]
        result.append([w[4 * t:4 * t + 4] for t in range(len(offsets))])
    print(json.dumps(result))


if __name__ == "__main__":
    main()
