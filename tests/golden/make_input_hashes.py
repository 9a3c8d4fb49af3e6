"""Writes input_hashes.txt: SHA-256 of generator output for the families
computed with exact arithmetic only (dyadic, uniform), so that any host
producing different input bytes is caught. Calls only ``synth_inputs``.

Run from the repository root:  python tests/golden/make_input_hashes.py
"""
import hashlib
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import synth_inputs as si  # noqa: E402

KEYS = [
    ("dyadic", "tf32", 256, 256, 0, "0"), ("dyadic", "tf32", 256, 256, 0, "1"),
    ("dyadic", "bf16", 128, 192, 100, "0"), ("dyadic", "fp16", 96, 64, 101, "1"),
    ("uniform", "tf32", 768, 768, 4, "0"), ("uniform", "bf16", 768, 768, 4, "1"),
    ("dyadic", "tf32", 64, 48, 102, "C"),
]

out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "input_hashes.txt")
with open(out, "w") as f:
    f.write("# family:dtype:RxC:seed:stream  sha256 of the row-major bytes\n")
    for fam, dt, r, c, seed, stream in KEYS:
        m = si.c_matrix(fam, r, c, seed) if stream == "C" else si.matrix(fam, dt, r, c, seed, int(stream))
        f.write(f"{fam}:{dt}:{r}x{c}:{seed}:{stream} {hashlib.sha256(m.tobytes()).hexdigest()}\n")
print("wrote", out)
