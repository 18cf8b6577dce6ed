"""Writes datagen_digests.txt: for the stream of each operand that the bench and
the tests draw, the SHA-256 of the storage bits of its first 4096 values, so
that a change to the generator, a distribution or a rounding step shows up as a
changed input rather than as a silent change of every measured workload.

Uniform streams use integer arithmetic and one exact scaling, so their digests
hold on any platform.  Box-Muller goes through log, cos and sin, which may
differ by an ulp between math libraries, so normal streams are recorded as
their first 32 values in fp64 (compared with a relative tolerance) instead.

Calls only the input generator.  Run from the repository root:
    python tests/golden/make_datagen_digests.py
"""
from __future__ import annotations

import hashlib
import math
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import datagen  # noqa: E402

N_VALUES = 4096
N_NORMAL = 32
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "datagen_digests.txt")

# (stream, seed, recipe): recipe is the storage the draw is rounded to
UNIFORM_STREAMS = [
    ("bf16 8192^3 + bias + GELU: A", 3001, "bf16/sqrt8192"),
    ("bf16 8192^3 + bias + GELU: B", 3002, "bf16/sqrt8192"),
    ("bf16 256^3: A", 1001, "bf16"),
    ("bf16 256^3: B", 1002, "bf16"),
    ("SGEMM 4096^3: A", 2001, "f32"),
    ("SGEMM 4096^3: B", 2002, "f32"),
    ("SGEMM 4096^3: C", 2003, "f32"),
    ("ragged 4097x3001x1000: A", 4001, "bf16"),
    ("ragged 4097x3001x1000: B", 4002, "bf16"),
    ("split-K 256x256x65536: A", 4011, "bf16"),
    ("split-K 256x256x65536: B", 4012, "bf16"),
    ("skinny 16x8192x8192: A", 4021, "bf16"),
    ("skinny 16x8192x8192: B", 4022, "bf16"),
    ("batched 64x1024^3: A", 5001, "bf16"),
    ("batched 64x1024^3: B", 5002, "bf16"),
]
NORMAL_STREAMS = [
    ("bf16 8192^3 + bias + GELU: bias", 3004),
    ("batched 64x1024^3: C", 5003),
]


def uniform_bits(seed: int, recipe: str) -> bytes:
    u = datagen.uniform(seed, (N_VALUES,))
    if recipe == "bf16/sqrt8192":
        # divided in fp64 as the bench does, then rounded once to bf16
        return datagen.to_bf16_bits(u / math.sqrt(8192)).astype("<u2").tobytes()
    if recipe == "bf16":
        return datagen.to_bf16_bits(u).astype("<u2").tobytes()
    if recipe == "f32":
        return datagen.to_f32(u).astype("<f4").tobytes()
    raise ValueError(recipe)


def main() -> None:
    lines = ["# SHA-256 of the storage bits (little-endian) of the first 4096 values of",
             "# each uniform operand stream, and the first 32 fp64 values of each normal",
             "# stream.  Written by tests/golden/make_datagen_digests.py (input generator",
             "# only).  Format: U|seed|recipe|sha256|name  or  N|seed|v0 v1 ...|name"]
    for name, seed, recipe in UNIFORM_STREAMS:
        digest = hashlib.sha256(uniform_bits(seed, recipe)).hexdigest()
        lines.append(f"U|{seed}|{recipe}|{digest}|{name}")
    for name, seed in NORMAL_STREAMS:
        vals = datagen.normal(seed, (N_NORMAL,))
        lines.append(f"N|{seed}|{' '.join(repr(float(v)) for v in vals)}|{name}")
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(f"wrote {OUT}")


if __name__ == "__main__":
    main()
